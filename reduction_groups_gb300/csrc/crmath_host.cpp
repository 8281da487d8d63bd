// Host build of the device exp / erf (crmath.cuh compiled as plain C++), for
// tests that check every tier element by element on the CPU.  Not part of the
// library's compute path: the kernels run the CUDA build of the same source.

#define PSK_HOST_BUILD 1
#include "crmath.cuh"

using namespace psk;

extern "C" {

// erf's Taylor tables as records (erf_record), built once
static const float* erf_records() {
  static float rec[12 * PSK_ERF_N32];
  static bool built = false;
  if (!built) {
    for (int i = 0; i < PSK_ERF_N32; ++i) erf_record(&psk_erf_p2[0][0], &psk_erf_h[0][0], i, rec + 12 * i);
    built = true;
  }
  return rec;
}

// which: 0 exp_cr, 1 erf_cr, 3 log_cr, 4 tanh_cr, 5 exp_fast,
// 6 erf_fast (signed),
// 10 erf tier 1 from the record tables (R; inputs in tier 1's range),
// 11 erf_fast of |x| from the record tables
void psk_host_unary(int which, const float* x, float* y, long n) {
  if (which == 10 || which == 11) {
    const float* rec = erf_records();
    for (long i = 0; i < n; ++i) {
      if (which == 11) {
        y[i] = erf_fast_abs_rec(fabsf(x[i]), rec);
      } else {
        float R, d;
        erf_tier1_core_rec(x[i], rec, R, d);
        y[i] = R;
      }
    }
    return;
  }
  for (long i = 0; i < n; ++i) {
    switch (which) {
      case 0: y[i] = exp_cr(x[i], psk_exp_tab2); break;
      case 1: y[i] = erf_cr(x[i], &psk_erf_p2[0][0], &psk_erf_h[0][0]); break;
      case 3: y[i] = log_cr(x[i], psk_log_tab); break;
      case 4: y[i] = tanh_cr(x[i], &psk_tanh_p2[0][0], &psk_tanh_h[0][0]); break;
      case 5: y[i] = exp_fast(x[i]); break;
      case 6: {
        const float a = fabsf(x[i]);
        const float r = a == a ? erf_fast_abs(a, &psk_erf_p2[0][0], &psk_erf_h[0][0]) : a;
        y[i] = copysignf(r, x[i]);
        break;
      }
      default: y[i] = NAN; break;
    }
  }
}

// Tier-by-tier: tier 1 with its decision flag (inputs must be in its range),
// tiers 2 and 3 on their own.  which: 0 exp, 1 erf, 2 log (normal positive
// x other than 1), 3 tanh (2^-12 <= x < its saturation).
void psk_host_tier(int which, int tier, const float* x, float* y, unsigned char* ok, long n) {
  for (long i = 0; i < n; ++i) {
    float r = 0.0f;
    bool k = true;
    if (which == 2) {
      if (tier == 1) {
        float d;
        log_tier1_core(x[i], 0, psk_log_tab, r, d);
        k = tier1_decided(r, d);
      } else {
        r = tier == 2 ? log_tier2(x[i]) : log_tier3(x[i], 0);
      }
    } else if (which == 3) {
      if (tier == 1) k = tanh_tier1(x[i], &psk_tanh_p2[0][0], &psk_tanh_h[0][0], r);
      else r = tier == 2 ? tanh_tier2(x[i]) : tanh_tier3(x[i]);
    } else if (tier == 1) {
      k = which == 0 ? exp_tier1(x[i], psk_exp_tab2, r)
                     : erf_tier1(x[i], &psk_erf_p2[0][0], &psk_erf_h[0][0], r);
    } else if (tier == 2) {
      r = which == 0 ? exp_tier2(x[i]) : erf_tier2(x[i]);
    } else {
      r = which == 0 ? exp_tier3(x[i]) : erf_tier3(x[i]);
    }
    y[i] = r;
    if (ok) ok[i] = k ? 1 : 0;
  }
}

// Tier-1 approximations before rounding, as binary64 (R + d) 2^n, to
// measure their error against a reference.  which: 0 exp, 1 erf, 2 log
// (normal positive x), 3 tanh.
void psk_host_tier1_value(int which, const float* x, double* y, long n) {
  for (long i = 0; i < n; ++i) {
    float R, d;
    if (which == 2) {
      log_tier1_core(x[i], 0, psk_log_tab, R, d);
      y[i] = (double)R + (double)d;
    } else if (which == 3) {
      tanh_tier1_core(x[i], &psk_tanh_p2[0][0], &psk_tanh_h[0][0], R, d);
      y[i] = (double)R + (double)d;
    } else if (which == 0) {
      int e;
      exp_tier1_core(x[i], psk_exp_tab2, R, d, e);
      y[i] = ldexp((double)R + (double)d, e);
    } else {
      erf_tier1_core(x[i], &psk_erf_p2[0][0], &psk_erf_h[0][0], R, d);
      y[i] = (double)R + (double)d;
    }
  }
}

// Division through the reciprocal against IEEE division, n random pairs
// drawn with a 64-bit LCG; returns the number of differing results.
long psk_host_div_check(unsigned long seed, long n, float a_lo_exp, float a_hi_exp, float b_hi) {
  unsigned long s = seed * 6364136223846793005ul + 1442695040888963407ul;
  long bad = 0;
  for (long i = 0; i < n; ++i) {
    s = s * 6364136223846793005ul + 1442695040888963407ul;
    uint32_t u1 = (uint32_t)(s >> 32);
    s = s * 6364136223846793005ul + 1442695040888963407ul;
    uint32_t u2 = (uint32_t)(s >> 32);
    // a: random sign-free mantissa and exponent in [a_lo_exp, a_hi_exp); b in [1, b_hi)
    float fa = ldexpf(1.0f + (float)(u1 & 0x7fffff) * 0x1p-23f,
                      (int)(a_lo_exp + (a_hi_exp - a_lo_exp) * ((u1 >> 23) / 512.0f)));
    float fb = 1.0f + (b_hi - 1.0f) * ((float)(u2 >> 8) * 0x1p-24f);
    volatile float ieee = fa / fb;
    float rb = 1.0f / fb;
    if (div_by_recip(fa, fb, rb) != ieee) ++bad;
  }
  return bad;
}


}  // extern "C"
