"""Pure-Python brute force of the sum collectives -- TEST INFRASTRUCTURE ONLY.

An independent second statement of the same definition, used on tiny inputs
to pin the C oracle bit for bit.  It shares nothing with ``oracle.c``: values
are decoded from the IEEE-754 field layouts by arithmetic on Python floats,
and every rounding is done by one generic value-level round-to-nearest-even
``round_ieee(x, precision, emin, emax)``.

Definition (standard collective API, MSCCL++ abstract point (3)): the sum over
ranks runs in order 0..N-1 from x_0, in binary32 for floating inputs (each
binary32 add is the exact sum rounded once; a binary64 add of two binary32
values followed by rounding to binary32 gives that same correctly rounded
result because 53 >= 2*24 + 2), then one rounding to the output format.
int32 wraps modulo 2^32.
"""
import math

INF = float("inf")

# (precision in bits incl. the implicit one, emin, emax)
FORMATS = {"fp32": (24, -126, 127), "bf16": (8, -126, 127), "fp16": (11, -14, 15)}


def _round_half_even(n):
    fl = math.floor(n)
    r = n - fl
    if r > 0.5 or (r == 0.5 and fl % 2 == 1):
        fl += 1
    return fl


def round_ieee(x, p, emin, emax):
    """Round a Python float to the binary format (p, emin, emax), ties to even."""
    if x != x or x in (INF, -INF) or x == 0.0:
        return x
    neg = x < 0
    a = -x if neg else x
    _, e = math.frexp(a)          # a in [2^(e-1), 2^e)
    binade = max(e - 1, emin)
    quantum = math.ldexp(1.0, binade - (p - 1))
    v = _round_half_even(a / quantum) * quantum
    # the largest finite value is (2 - 2^(1-p)) * 2^emax; anything rounding past it overflows
    if v >= math.ldexp(1.0, emax + 1):
        v = INF
    return -v if neg else v


def decode(bits, dtype):
    """Raw storage -> Python float (or int for int32)."""
    if dtype == "int32":
        return int(bits)
    if dtype == "fp32":
        return float(bits)  # numpy float32 -> exact double
    b = int(bits) & 0xFFFF
    if dtype == "bf16":
        sign, e, m, mbits, bias = b >> 15, (b >> 7) & 0xFF, b & 0x7F, 7, 127
        emax_field = 0xFF
    else:
        sign, e, m, mbits, bias = b >> 15, (b >> 10) & 0x1F, b & 0x3FF, 10, 15
        emax_field = 0x1F
    if e == emax_field:
        v = INF if m == 0 else float("nan")
    elif e == 0:
        v = math.ldexp(m, 1 - bias - mbits)
    else:
        v = math.ldexp((1 << mbits) + m, e - bias - mbits)
    return -v if sign else v


def encode(v, dtype):
    """Python float already representable in ``dtype`` -> raw storage bits / value."""
    if dtype == "fp32":
        return v
    if v != v:
        return None  # NaN: callers compare NaN-ness only
    neg = math.copysign(1.0, v) < 0
    a = abs(v)
    if dtype == "bf16":
        mbits, bias, efield = 7, 127, 0xFF
    else:
        mbits, bias, efield = 10, 15, 0x1F
    if a == INF:
        bits = efield << mbits
    elif a == 0.0:
        bits = 0
    else:
        _, e = math.frexp(a)
        E = e - 1
        emin = 1 - bias
        if E < emin:
            bits = int(a / math.ldexp(1.0, emin - mbits))
        else:
            frac = a / math.ldexp(1.0, E) - 1.0
            bits = ((E + bias) << mbits) | int(round(frac * (1 << mbits)))
    return bits | (0x8000 if neg else 0)


def _max_ieee(a, b):
    """IEEE 754-2019 maximum of two Python floats: NaN wins, -0 < +0."""
    if a != a or b != b:
        return float("nan")
    if a == b:
        return b if math.copysign(1.0, a) < 0 else a
    return a if a > b else b


def _min_ieee(a, b):
    if a != a or b != b:
        return float("nan")
    if a == b:
        return a if math.copysign(1.0, a) < 0 else b
    return a if a < b else b


def allreduce_op_elem(values, dtype, op):
    """MAX / MIN over ranks in order 0..N-1 of the decoded values; int32 as integers."""
    if dtype == "int32":
        vals = [int(v) for v in values]
        return max(vals) if op == "max" else min(vals)
    f = _max_ieee if op == "max" else _min_ieee
    acc = decode(values[0], dtype)
    for v in values[1:]:
        acc = f(acc, decode(v, dtype))
    return acc


def allreduce_op(xs, dtype, op):
    n = len(xs[0])
    return [allreduce_op_elem([x[i] for x in xs], dtype, op) for i in range(n)]


def allreduce_elem(values, dtype):
    """One output element from the N ranks' raw values at that index."""
    if dtype == "int32":
        s = sum(int(v) for v in values)
        return ((s + 2 ** 31) % 2 ** 32) - 2 ** 31
    p, emin, emax = FORMATS["fp32"]
    acc = decode(values[0], dtype)
    for v in values[1:]:
        acc = round_ieee(acc + decode(v, dtype), p, emin, emax)
    if dtype == "fp32":
        return acc
    return round_ieee(acc, *FORMATS[dtype])


def allreduce(xs, dtype):
    """List of per-element results (Python floats / ints) for rank buffers xs."""
    n = len(xs[0])
    return [allreduce_elem([x[i] for x in xs], dtype) for i in range(n)]


def reduce_scatter(xs, dtype, rank, m):
    return [allreduce_elem([x[rank * m + j] for x in xs], dtype) for j in range(m)]


def allgather(xs):
    out = []
    for x in xs:
        out.extend(list(x))
    return out


def ring_barrier_counts(n, iters):
    """Simulate the token: per iteration rank r signals (r+1) mod N once."""
    counts = [[0] * n for _ in range(n)]
    for _ in range(iters):
        holder = 0
        for _hop in range(n):
            nxt = (holder + 1) % n
            counts[nxt][holder] += 1
            holder = nxt
    return counts
