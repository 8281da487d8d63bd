"""Writes crmath_tables.inc: the constant tables of the device exp / erf /
log / tanh.

Run by hand (needs mpmath, 300-bit arithmetic); the generated file is
committed, so building the library does not need mpmath.

  python gen_crmath_tables.py > crmath_tables.inc

Tables:
* exp: 2^(j/1024), j = 0..1023, as float pairs (hi, lo interleaved) for the
  binary32 path and 2^(j/32), j = 0..31, as binary64 values for the binary64
  path; the Cody-Waite pieces of ln2/1024 and ln2/32.
* erf: Taylor polynomials of erf about interval centres c, with
  coefficients erf^(k)(c)/k! = (2/sqrt(pi)) (-1)^(k-1) H_{k-1}(c) exp(-c^2)/k!
  (k >= 1, H the physicists' Hermite polynomials) and coefficient 0 equal to
  erf(c).  The binary32 path uses 128 intervals of width 1/32 centred at
  i/32 (interval 0 is [0, 1/64]), coefficients 0..3 as float pairs (hi, lo
  interleaved) and 4..D32 as floats, D32 the least degree whose truncation
  stays below 2^-48 relative on every interval; the binary64 path uses 32
  intervals of width 1/8 centred at i/8, degree 12 (below 2^-61).
* tanh: Taylor polynomials about c = i/32 in the erf layout (width 1/32,
  coefficients 0..3 as float pairs, the rest as floats), up to the least
  binary32 from which tanh rounds to 1; coefficient k is P_k(tanh c)/k! with
  P_0(T) = T and P_{k+1}(T) = (1 - T^2) P_k'(T) (d tanh/dx = 1 - tanh^2).
* log: 512 intervals by the top nine significand bits of x, each with
  c (a multiple of 2^-10 near 1/m, exactly 1 and 1/2 on the two intervals
  touching m = 1 and m = 2), s (1 where the interval lies above sqrt 2: the
  significand is then read as m/2 and the exponent as e + 1) and
  T = -log(c 2^s) as a float pair, stored as (c, T hi, T lo, s); r = m c - 1
  is exact in binary32 (checked) and below 2^-9 in magnitude.
"""

import mpmath as mp

mp.mp.prec = 300

N_INT = 32          # binary64 path: intervals of width 1/8
N_INT32 = 128       # binary32 path: intervals of width 1/32
W32 = mp.mpf(1) / 32
N_PAIR = 4          # binary32 path: coefficients 0..N_PAIR-1 as float pairs
D64 = 12


def rn(x, bits):
    with mp.workprec(bits):
        return +mp.mpf(x)


def f32(x):
    v = rn(x, 24)
    return float(v)


def f64(x):
    return float(rn(x, 53))


def split_f32(x):
    hi = rn(x, 24)
    lo = rn(mp.mpf(x) - hi, 24)
    return float(hi), float(lo)


def trunc_bits(x, bits):
    """x truncated (towards zero) to `bits` significant bits."""
    m, e = mp.frexp(x)
    scale = mp.mpf(2) ** bits
    return mp.ldexp(mp.floor(abs(m) * scale) * mp.sign(m) / scale, e)


def fmt32(v):
    return f"{float(v).hex()}f" if v != 0 else "0.0f"


def fmt64(v):
    return float(v).hex() if v != 0 else "0.0"


def taylor(c, D):
    """erf Taylor coefficients about c, degree D (exact, high precision)."""
    cs = [mp.erf(c)]
    e = 2 / mp.sqrt(mp.pi) * mp.exp(-c * c)
    for k in range(1, D + 1):
        cs.append(e * (-1) ** (k - 1) * mp.hermite(k - 1, c) / mp.factorial(k))
    return cs


def degree32():
    """Least degree D with |sum_{k>D} c_k t^k| < 2^-48 erf(c + t) on every
    binary32 interval (|t| <= 1/64; t >= 0 on interval 0), the tail bounded by
    twice its first two terms (the coefficients shrink geometrically)."""
    for D in range(5, 16):
        ok = True
        for i in range(N_INT32):
            c = i * W32
            cs = taylor(c, D + 2)
            h = W32 / 2
            lo_a = c - h if i > 0 else mp.mpf(2) ** -60
            tail = 2 * (abs(cs[D + 1]) * h ** (D + 1) + abs(cs[D + 2]) * h ** (D + 2))
            if i == 0:   # erf(t) ~ 1.128 t: compare the tail's t-power with t
                tail = 2 * (abs(cs[D + 1]) * h ** D + abs(cs[D + 2]) * h ** (D + 1)) * h
                lo_a = h
            if tail >= mp.mpf(2) ** -48 * mp.erf(lo_a):
                ok = False
                break
        if ok:
            return D
    raise AssertionError("no degree below 16")


def check_fast2sum(c32hi, D32):
    """The binary32 evaluation adds t*V_{k+1} to coefficient k (k = 3, 2, 1, 0)
    with Fast2Sum, which is exact when the coefficient is 0 or not smaller in
    magnitude; check that bound over each interval."""
    for i in range(N_INT32):
        ts = [mp.mpf(j) / 4096 for j in range(0, 65)] if i == 0 else \
             [mp.mpf(j) / 4096 for j in range(-64, 65)]
        for t in ts:
            v = mp.mpf(0)
            for k in range(D32, -1, -1):
                tv = t * v
                if k <= N_PAIR - 1:
                    ck = mp.mpf(c32hi[k][i])
                    assert ck == 0 or abs(ck) >= abs(tv) * 2, (i, k, float(t))
                v = mp.mpf(c32hi[k][i]) + tv


def fast2sum_failures(hi, npair, n_int, factor, t_lo0):
    """The pair steps k (0..npair-1) at which Fast2Sum's exact condition
    |c_k| >= |t V_{k+1}| (times `factor`) or c_k = 0 fails on some interval of
    a table of n_int intervals (interval 0 starting at t_lo0); those steps
    add with the branch-free TwoSum instead, which is exact in any order."""
    D = len(hi) - 1
    bad = set()
    for i in range(n_int):
        ts = [mp.mpf(j) / 4096 for j in range(0, 65)] if i == 0 else \
             [mp.mpf(j) / 4096 for j in range(-64, 65)]
        if i == 0:
            ts = [max(t, t_lo0) for t in ts]
        for t in ts:
            v = mp.mpf(0)
            for k in range(D, -1, -1):
                tv = t * v
                if k <= npair - 1:
                    ck = mp.mpf(hi[k][i])
                    if not (ck == 0 or abs(ck) >= abs(tv) * factor):
                        bad.add(k)
                v = mp.mpf(hi[k][i]) + tv
    return bad


def tanh_taylor(c, D):
    """tanh Taylor coefficients about c through degree D (integer derivative
    polynomials evaluated at tanh c)."""
    T = mp.tanh(c)
    poly = [0, 1]                       # P_0(T) = T, coefficients by power
    out = [T]
    for k in range(1, D + 1):
        der = [j * poly[j] for j in range(1, len(poly))]            # P'
        nxt = [0] * (len(der) + 2)
        for j, a in enumerate(der):                                 # (1 - T^2) P'
            nxt[j] += a
            nxt[j + 2] -= a
        poly = nxt
        val = mp.mpf(0)
        for a in reversed(poly):
            val = val * T + a
        out.append(val / mp.factorial(k))
    return out


def tanh_one_from():
    """Least binary32 a with RN(tanh a) = 1, i.e. 1 - tanh(a) <= 2^-25."""
    import struct
    nxt = lambda v, d: struct.unpack("f", struct.pack("I", struct.unpack("I", struct.pack("f", v))[0] + d))[0]
    done = lambda a: 1 - mp.tanh(a) <= mp.mpf(2) ** -25
    a = struct.unpack("f", struct.pack("f", float(mp.atanh(1 - mp.mpf(2) ** -25))))[0]
    while not done(a):
        a = nxt(a, 1)
    while done(nxt(a, -1)):
        a = nxt(a, -1)
    return a


TANH_LO = mp.mpf(2) ** -12     # below, tanh(a) rounds to a


def tanh_degree(n_int):
    for D in range(5, 16):
        ok = True
        for i in range(n_int):
            c = i * W32
            cs = tanh_taylor(c, D + 2)
            h = W32 / 2
            if i == 0:
                tail = 2 * (abs(cs[D + 1]) * h ** D + abs(cs[D + 2]) * h ** (D + 1)) * h
                lo_a = h
            else:
                tail = 2 * (abs(cs[D + 1]) * h ** (D + 1) + abs(cs[D + 2]) * h ** (D + 2))
                lo_a = c - h
            if tail >= mp.mpf(2) ** -48 * mp.tanh(lo_a):
                ok = False
                break
        if ok:
            return D
    raise AssertionError("no degree below 16")


def log_table():
    """(c, T hi, T lo, s) per interval, the largest |r|, and checks."""
    rows = []
    rmax = mp.mpf(0)
    sqrt2 = mp.sqrt(2)
    for i in range(512):
        m_lo = 1 + mp.mpf(i) / 512
        m_hi = 1 + mp.mpf(i + 1) / 512 - mp.mpf(2) ** -23     # last binary32 in the interval
        mid = 1 + (mp.mpf(i) + mp.mpf(0.5)) / 512
        s = 1 if mid > sqrt2 else 0
        if i == 0:
            c = mp.mpf(1)
        elif i == 511:
            c = mp.mpf(1) / 2
        else:
            c = mp.nint(1024 / mid) / 1024
        rloc = mp.mpf(0)
        for m in (m_lo, m_hi):
            r = m * c - 1
            # exact in binary32: a multiple of 2^-33 below 2^-9 (24 bits)
            assert abs(r) < mp.mpf(2) ** -9, (i, float(r))
            assert mp.floor(r * 2 ** 33) == r * 2 ** 33
            rloc = max(rloc, abs(r))
        rmax = max(rmax, rloc)
        T = -mp.log(c * 2 ** s)
        th, tl = split_f32(T)
        # T hi + r is added by Fast2Sum: T = 0 or |T hi| >= |r|
        assert th == 0 or abs(th) >= rloc, (i, th, float(rloc))
        rows.append((float(c), th, tl, float(s)))
    return rows, rmax


def main():
    out = []
    w = out.append
    w("// Generated by gen_crmath_tables.py -- do not edit.")
    ln2_32 = mp.log(2) / 32
    ln2_n = mp.log(2) / 1024
    # binary32 reduction by ln2/1024, |k| < 2^17 (|x| <= 87): L1 = RN(ln2/1024)
    # (x - k L1 is exact: a multiple of 2^-35 below 2^-11); L2 carries 7
    # significant bits (k L2 exact); L3 the rest, rounded.  |k (ln2/1024 - L1)|
    # stays below 2^-21.99.
    L1 = rn(ln2_n, 24)
    L2 = trunc_bits(ln2_n - L1, 7)
    L3 = rn(ln2_n - L1 - L2, 24)
    assert mp.mpf(2) ** -11 <= L1 < mp.mpf(2) ** -10
    assert 128526 * abs(ln2_n - L1) < mp.mpf(2) ** -21.99   # |k| <= 128526 for |x| <= 87
    w(f"#define PSK_EXP_TAB_N 1024")
    w(f"#define PSK_EXP_INV_L {fmt32(f32(1024 / mp.log(2)))}")
    w(f"#define PSK_EXP_L1 {fmt32(L1)}")
    w(f"#define PSK_EXP_L2 {fmt32(L2)}")
    w(f"#define PSK_EXP_L3 {fmt32(L3)}")
    # binary64 Cody-Waite: |k| < 2^13, L1 carries 40 significant bits
    L1d = trunc_bits(ln2_32, 40)
    L2d = rn(ln2_32 - L1d, 53)
    w(f"#define PSK_EXP_INV_LD {fmt64(f64(32 / mp.log(2)))}")
    w(f"#define PSK_EXP_L1D {fmt64(L1d)}")
    w(f"#define PSK_EXP_L2D {fmt64(L2d)}")
    w(f"#define PSK_TWO_OVER_SQRTPI_D {fmt64(f64(2 / mp.sqrt(mp.pi)))}")
    # double-double constants of the last tier
    for name, val in (("LN2", mp.log(2)), ("TWO_OVER_SQRTPI", 2 / mp.sqrt(mp.pi))):
        hi = rn(val, 53)
        lo = rn(val - hi, 53)
        w(f"#define PSK_DD_{name}_HI {fmt64(hi)}")
        w(f"#define PSK_DD_{name}_LO {fmt64(lo)}")
    w(f"#define PSK_DD_INV_LN2 {fmt64(f64(1 / mp.log(2)))}")
    w(f"#define PSK_INV_SQRT2 {fmt32(f32(1 / mp.sqrt(2)))}   // gelu's RN_f32(1/sqrt 2)")
    # faithful binary32 exp: k = rint(x / ln2), |k| < 2^8, ln2 hi carries 16 bits
    h16 = trunc_bits(mp.log(2), 16)
    w(f"#define PSK_FEXP_INV_LN2 {fmt32(f32(1 / mp.log(2)))}")
    w(f"#define PSK_FEXP_LN2_HI {fmt32(h16)}")
    w(f"#define PSK_FEXP_LN2_LO {fmt32(f32(mp.log(2) - h16))}")
    pairs = [split_f32(mp.mpf(2) ** (mp.mpf(j) / 1024)) for j in range(1024)]
    w("PSK_GTAB float psk_exp_tab2[2048] = {")
    for j0 in range(0, 1024, 4):
        w("  " + ", ".join(f"{fmt32(h)}, {fmt32(l)}" for h, l in pairs[j0:j0 + 4]) + ",")
    w("};")
    w("PSK_TAB double psk_exp_tab_d[32] = {" +
      ", ".join(fmt64(f64(mp.mpf(2) ** (mp.mpf(j) / 32))) for j in range(32)) + "};")

    # erf, binary32 path: [coefficient][interval] so that lanes reading
    # different intervals hit different shared-memory banks.
    D32 = degree32()
    c32hi = [[0.0] * N_INT32 for _ in range(D32 + 1)]
    c32lo = [[0.0] * N_INT32 for _ in range(N_PAIR)]
    for i in range(N_INT32):
        t32 = taylor(i * W32, D32)
        for k in range(D32 + 1):
            if k < N_PAIR:
                c32hi[k][i], c32lo[k][i] = split_f32(t32[k])
            else:
                c32hi[k][i] = f32(t32[k])
    check_fast2sum(c32hi, D32)
    c64 = [[0.0] * N_INT for _ in range(D64 + 1)]
    for i in range(N_INT):
        t64 = taylor(mp.mpf(i) / 8, D64)
        for k in range(D64 + 1):
            c64[k][i] = f64(t64[k])
    # smallest binary32 a with erfc(a) < 2^-25: from there on erf rounds to 1
    import struct
    root = mp.findroot(lambda a: mp.erfc(a) - mp.mpf(2) ** -25, 3.9)
    a = struct.unpack("f", struct.pack("f", float(root)))[0]
    nxt = lambda v, d: struct.unpack("f", struct.pack("I", struct.unpack("I", struct.pack("f", v))[0] + d))[0]
    while mp.erfc(a) >= mp.mpf(2) ** -25:
        a = nxt(a, 1)
    while mp.erfc(nxt(a, -1)) < mp.mpf(2) ** -25:
        a = nxt(a, -1)
    w(f"#define PSK_ERF_ONE_FROM {fmt32(a)}")
    w(f"#define PSK_ERF_N32 {N_INT32}")
    w(f"#define PSK_ERF_D32 {D32}")
    w(f"#define PSK_ERF_D64 {D64}")
    w(f"#define PSK_ERF_NPAIR {N_PAIR}")
    w(f"PSK_GTAB float psk_erf_p2[{N_PAIR}][{2 * N_INT32}] = {{   // coefficients 0..{N_PAIR - 1}: (hi, lo) per interval")
    for k in range(N_PAIR):
        w("  {" + ", ".join(f"{fmt32(c32hi[k][i])}, {fmt32(c32lo[k][i])}" for i in range(N_INT32)) + "},")
    w("};")
    w(f"PSK_GTAB float psk_erf_h[{D32 + 1 - N_PAIR}][{N_INT32}] = {{   // coefficients {N_PAIR}..{D32}")
    for k in range(N_PAIR, D32 + 1):
        w("  {" + ", ".join(fmt32(v) for v in c32hi[k]) + "},")
    w("};")
    w(f"PSK_TAB double psk_erf_c64[{D64 + 1}][32] = {{")
    for k in range(D64 + 1):
        w("  {" + ", ".join(fmt64(v) for v in c64[k]) + "},")
    w("};")

    # tanh, binary32 path: the erf layout over [0, tanh's saturation point]
    one = tanh_one_from()
    n_t = int(mp.nint(mp.mpf(one) * 32)) + 1
    Dt = tanh_degree(n_t)
    thi = [[0.0] * n_t for _ in range(Dt + 1)]
    tlo = [[0.0] * n_t for _ in range(N_PAIR)]
    for i in range(n_t):
        tc = tanh_taylor(i * W32, Dt)
        for k in range(Dt + 1):
            if k < N_PAIR:
                thi[k][i], tlo[k][i] = split_f32(tc[k])
            else:
                thi[k][i] = f32(tc[k])
    bad = fast2sum_failures(thi, N_PAIR, n_t, mp.mpf(1.001), TANH_LO)
    w(f"#define PSK_TANH_ONE_FROM {fmt32(one)}")
    w(f"#define PSK_TANH_TWOSUM_MASK {sum(1 << k for k in bad)}   // pair steps added with TwoSum")
    w(f"#define PSK_TANH_N32 {n_t}")
    w(f"#define PSK_TANH_D32 {Dt}")
    w(f"PSK_GTAB float psk_tanh_p2[{N_PAIR}][{2 * n_t}] = {{   // coefficients 0..{N_PAIR - 1}: (hi, lo) per interval")
    for k in range(N_PAIR):
        w("  {" + ", ".join(f"{fmt32(thi[k][i])}, {fmt32(tlo[k][i])}" for i in range(n_t)) + "},")
    w("};")
    w(f"PSK_GTAB float psk_tanh_h[{Dt + 1 - N_PAIR}][{n_t}] = {{   // coefficients {N_PAIR}..{Dt}")
    for k in range(N_PAIR, Dt + 1):
        w("  {" + ", ".join(fmt32(v) for v in thi[k]) + "},")
    w("};")

    # log, binary32 path.  e' ln2 = e' L1 + e' L2 + e' L3: L1 and L2 carry
    # 16 significant bits each, so e' L1 and e' L2 are exact for |e'| < 2^8.
    ln2 = mp.log(2)
    L1 = trunc_bits(ln2, 16)
    L2 = trunc_bits(ln2 - L1, 16)
    L3 = rn(ln2 - L1 - L2, 24)
    w(f"#define PSK_LOG_L1 {fmt32(L1)}")
    w(f"#define PSK_LOG_L2 {fmt32(L2)}")
    w(f"#define PSK_LOG_L3 {fmt32(L3)}")
    rows, rmax = log_table()
    w(f"// largest |r| = 2^{float(mp.log(rmax, 2)):.3f}")
    w("PSK_GTAB float psk_log_tab[2048] = {   // per interval: c, T hi, T lo, s")
    for i0 in range(0, 512, 2):
        w("  " + ", ".join(", ".join(fmt32(v) for v in rows[i]) for i in (i0, i0 + 1)) + ",")
    w("};")
    print("\n".join(out))


if __name__ == "__main__":
    main()
