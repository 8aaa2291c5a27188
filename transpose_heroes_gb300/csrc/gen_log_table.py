"""Generate log_table.inc, the tables of the correctly rounded f32 log used by the CUDA kernels.

Method (table-driven logarithm in the style of P. T. P. Tang, "Table-driven implementation of the
logarithm function in IEEE floating-point arithmetic", ACM TOMS 16(4), 1990):

  x = 2^e * m with m in [OFF, 2*OFF), OFF ~ 0.706 (so that log m is small on both sides of 1);
  interval i of m (the 8 mantissa bits of bits(x) - bits(OFF) below the exponent) has a centre c_i;
  log x = e*ln2 + log(c_i) + log1p(r),  r = m * inv_c - 1,  inv_c ~ 1/c_i.

inv_c is chosen on a power-of-two grid coarse enough that r = fma(m, inv_c, -1) is EXACT in f32 for
every m of its interval (checked exhaustively below); log(c) = -log(inv_c) is then stored as an
unevaluated f32 pair (hi, lo), and e*ln2 as a pair per exponent. The interval holding 1.0 has
inv_c = 1, so log x = log1p(x - 1) near 1 with no cancellation. For the intervals with e = 0 the
generator also checks |log c_hi| >= max |r| over the interval, which the kernel's Fast2Sum relies on.

All values are computed with Python's decimal module at 60 digits and rounded to f32 exactly. The
accurate stage also gets log(c) and ln 2 as double-doubles (each part rounded to double exactly).
A second, 32-entry table serves a cheap first pass (error ~2^-32, see cr_log.cuh): its interval holding
1.0 is centred on 1.0 as well, and log(c) hi is rounded to a multiple of 2^-16 so that
e*LN2_A + log(c)_hi is exact in f32 for every exponent (LN2_A = ln2 rounded to 16 bits; Tang's device);
log(c)_lo = log(c) - log(c)_hi and LN2_B = ln2 - LN2_A are single floats. The generator checks that
r is exact and that |log(c)_hi| >= max |r| wherever c != 1 (Fast2Sum precondition).

Run:  python gen_log_table.py  (writes log_table.inc next to this file).
"""

from __future__ import annotations

import os
import struct
from decimal import Decimal, getcontext

import numpy as np

getcontext().prec = 60

OFF = 0x3F34C000       # bits of ~0.70605; 1.0 sits at the centre of its interval
INDEX_BITS = 8
SHIFT = 23 - INDEX_BITS
N = 1 << INDEX_BITS
E_MIN, E_MAX = -150, 129  # covers subnormals (scaled by 2^23 first) up to the largest finite f32


def f32_of_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def bits_of_f32(f: float) -> int:
    return struct.unpack("<I", struct.pack("<f", f))[0]


def round_f32(d: Decimal) -> float:
    """Nearest f32 to the Decimal d (ties to even), decided exactly."""
    f = np.float32(float(d))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        dist = abs(Decimal(float(cand)) - d)
        key = (dist, bits_of_f32(float(cand)) & 1)
        if best is None or key < best[0]:
            best = (key, float(cand))
    return best[1]


def split(d: Decimal):
    hi = round_f32(d)
    lo = round_f32(d - Decimal(hi))
    return hi, lo


def interval_values(i: int) -> np.ndarray:
    lo = OFF + (i << SHIFT)
    bits = np.arange(lo, lo + (1 << SHIFT), dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32).astype(np.float64)


def residual_exact(m: np.ndarray, inv_c: float) -> tuple[bool, float]:
    prod = m * inv_c                   # exact in f64: 24 + few bits
    r = prod - 1.0                     # exact in f64
    ok = bool(np.all(r.astype(np.float32).astype(np.float64) == r))
    return ok, float(np.max(np.abs(r)))


def build():
    ln2 = Decimal(2).ln()
    ctab = []
    max_r = 0.0
    for i in range(N):
        m = interval_values(i)
        if m[0] <= 1.0 <= m[-1]:
            inv_c, q = 1.0, None
            ok, mr = residual_exact(m, inv_c)
            assert ok
        else:
            target = 2.0 / (m[0] + m[-1])
            chosen = None
            for q in range(14, 0, -1):
                cand = round(target * 2 ** q) / 2 ** q
                ok, mr = residual_exact(m, cand)
                if ok:
                    chosen = (cand, mr)
                    break
            assert chosen is not None, i
            inv_c, mr = chosen
        logc = -Decimal(inv_c).ln()
        hi, lo = split(logc)
        if inv_c != 1.0:
            assert abs(hi) >= mr, (i, hi, mr)  # Fast2Sum(log c_hi, r) precondition for e = 0
        max_r = max(max_r, mr)
        ctab.append((inv_c, hi, lo, mr))
    etab = []
    for e in range(E_MIN, E_MAX + 1):
        hi, lo = split(Decimal(e) * ln2)
        etab.append((hi, lo))
    return ctab, etab, max_r


# cheap first-pass table: 32 intervals
OFF1_TARGET = 0x3F3504F3
INDEX_BITS1 = 5
SHIFT1 = 23 - INDEX_BITS1


def off1():
    half = 1 << (SHIFT1 - 1)
    cands = [o for o in range(0x3F300000, 0x3F3A0000) if (0x3F800000 - o) % (1 << SHIFT1) == half]
    return min(cands, key=lambda o: abs(o - OFF1_TARGET))


def build1():
    ln2 = Decimal(2).ln()
    ln2_a = Decimal(round(ln2 * 2 ** 16)) / 2 ** 16
    ln2_b = round_f32(ln2 - ln2_a)
    off = off1()
    rows = []
    max_r = 0.0
    for i in range(1 << INDEX_BITS1):
        lo = off + (i << SHIFT1)
        bits = np.arange(lo, lo + (1 << SHIFT1), dtype=np.uint64).astype(np.uint32)
        m = bits.view(np.float32).astype(np.float64)
        if m[0] <= 1.0 <= m[-1]:
            inv_c = 1.0
            ok, mr = residual_exact(m, inv_c)
            assert ok
        else:
            target = 2.0 / (m[0] + m[-1])
            chosen = None
            for q in range(14, 0, -1):
                cand = round(target * 2 ** q) / 2 ** q
                ok, mr = residual_exact(m, cand)
                if ok:
                    chosen = (cand, mr)
                    break
            assert chosen is not None
            inv_c, mr = chosen
        logc = -Decimal(inv_c).ln()
        hi = Decimal(round(logc * 2 ** 16)) / 2 ** 16
        assert float(hi) == round_f32(hi)  # 16-bit grid value is an exact f32
        lo_ = round_f32(logc - hi)
        if inv_c != 1.0:
            assert abs(float(hi)) >= mr, (i, hi, mr)
        max_r = max(max_r, mr)
        rows.append((inv_c, float(hi), lo_))
    return off, float(ln2_a), ln2_b, rows, max_r


def round_f64(d: Decimal) -> float:
    """Nearest double to the Decimal d (ties to even), decided exactly."""
    f = float(d)
    best = None
    for cand in (np.nextafter(f, -np.inf), f, np.nextafter(f, np.inf)):
        dist = abs(Decimal(float(cand)) - d)
        key = (dist, struct.unpack("<Q", struct.pack("<d", float(cand)))[0] & 1)
        if best is None or key < best[0]:
            best = (key, float(cand))
    return best[1]


def split_dd(d: Decimal):
    hi = round_f64(d)
    lo = round_f64(d - Decimal(hi))
    return hi, lo


def fmt(v: float) -> str:
    return f"{float(v).hex()}f" if v != 0 else "0.0f"


def main():
    ctab, etab, max_r = build()
    here = os.path.dirname(os.path.abspath(__file__))
    out = os.path.join(here, "log_table.inc")
    with open(out, "w") as f:
        f.write("// Generated by gen_log_table.py -- do not edit. Tables of the correctly rounded f32 log.\n")
        f.write(f"// Intervals: {N} (index = bits 15..22 of bits(x) - 0x{OFF:08X}); max |r| = {max_r!r}\n")
        f.write(f"#define HLO_LOG_OFF 0x{OFF:08X}u\n")
        f.write(f"#define HLO_LOG_SHIFT {SHIFT}\n")
        f.write(f"#define HLO_LOG_NC {N}\n")
        f.write(f"#define HLO_LOG_EMIN ({E_MIN})\n")
        f.write(f"#define HLO_LOG_NE {len(etab)}\n")
        f.write("// {inv_c, log(c) hi, log(c) lo, max |r| on the interval}\n")
        f.write("static __device__ const float4 kLogCTab[HLO_LOG_NC] = {\n")
        for row in ctab:
            f.write("  {" + ", ".join(fmt(v) for v in row) + "},\n")
        f.write("};\n")
        f.write("// {e*ln2 hi, e*ln2 lo} for e = HLO_LOG_EMIN ...\n")
        f.write("static __device__ const float2 kLogETab[HLO_LOG_NE] = {\n")
        for row in etab:
            f.write("  {" + ", ".join(fmt(v) for v in row) + "},\n")
        f.write("};\n")
        # accurate stage: log(c) = hi + lo with hi on the 2^-45 grid, ln 2 = hi + lo with hi on the 2^-44
        # grid, so that e*LN2_HI + LOGC_HI is exact in double for every |e| <= 149 (a multiple of 2^-45
        # below 2^7: 52 bits)
        f.write("// log(c) = -log(inv_c) as {hi on the 2^-45 grid, lo = RN(log(c) - hi)} (accurate stage)\n")
        f.write("static __device__ const double2 kLogC3[HLO_LOG_NC] = {\n")
        for row in ctab:
            logc = -Decimal(row[0]).ln()
            hi = Decimal(round(logc * 2 ** 45)) / 2 ** 45
            assert float(hi) == hi
            lo = round_f64(logc - hi)
            f.write(f"  {{{float(hi).hex()}, {lo.hex() if lo != 0 else '0.0'}}},\n")
        f.write("};\n")
        ln2 = Decimal(2).ln()
        ln2_hi = Decimal(round(ln2 * 2 ** 44)) / 2 ** 44
        assert float(ln2_hi) == ln2_hi
        ln2_lo = round_f64(ln2 - ln2_hi)
        f.write(f"#define HLO_LN2_DD_HI {float(ln2_hi).hex()}\n#define HLO_LN2_DD_LO {ln2_lo.hex()}\n")
        off, ln2_a, ln2_b, rows, max_r1 = build1()
        f.write(f"// First-pass table: 32 intervals (index = bits {SHIFT1}..22 of bits(x) - 0x{off:08X}); max |r| = {max_r1!r}\n")
        f.write(f"#define HLO_LOG1_OFF 0x{off:08X}u\n")
        f.write(f"#define HLO_LOG1_SHIFT {SHIFT1}\n")
        f.write(f"#define HLO_LOG1_LN2_A {fmt(ln2_a)}\n")
        f.write(f"#define HLO_LOG1_LN2_B {fmt(ln2_b)}\n")
        for name, col in (("kLog1Inv", 0), ("kLog1Hi", 1), ("kLog1Lo", 2)):
            f.write(f"static __device__ const float {name}[32] = {{" + ", ".join(fmt(r[col]) for r in rows) + "};\n")
    print(f"wrote {out}; max |r| = {max_r} (2^{np.log2(max_r):.2f}); first pass max |r| = 2^{np.log2(max_r1):.2f}")


if __name__ == "__main__":
    main()
