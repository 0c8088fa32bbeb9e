// Streaming numeric conversion of one field's value bytes (ParPaRaw Section
// 3.3, "converting the symbol string to the column's type"; Section 4.3,
// "the empty string is parsed as the column's default value").
//
// Integers: grammar [+-]?[0-9]+, exact, range-checked per column type.
// Floats: grammar [+-]?([0-9]+(\.[0-9]*)?|\.[0-9]+)([eE][+-]?[0-9]+)?.
//   Fast path (Clinger, "How to read floating point numbers accurately",
//   PLDI 1990): a significand of at most 2^53 and |e10| <= 22 gives the
//   correctly rounded result with one exact-operand multiply or divide.
//   Otherwise the first 19 significant digits are scaled by 10^e10 in
//   double-double arithmetic (Dekker's exact product via FMA, fast two-sum)
//   against a table of 10^k computed exactly, and rounded once: the result
//   is within 1 ulp of the correctly rounded value.
#pragma once
#include <cstdint>
#include "pp.h"
#include "pow10_table.inc"

namespace ppn {

// 1e0 .. 1e22 are exactly representable in binary64
__device__ __forceinline__ double exact_pow10(int k) {
  constexpr double T[23] = {1e0,  1e1,  1e2,  1e3,  1e4,  1e5,  1e6,  1e7,
                            1e8,  1e9,  1e10, 1e11, 1e12, 1e13, 1e14, 1e15,
                            1e16, 1e17, 1e18, 1e19, 1e20, 1e21, 1e22};
  return T[k];
}

struct DD { double hi, lo; };
__device__ __forceinline__ DD dd_mul(DD a, DD b) {
  double p = a.hi * b.hi;
  double e = fma(a.hi, b.hi, -p);          // exact low part of a.hi*b.hi
  e = fma(a.hi, b.lo, e);
  e = fma(a.lo, b.hi, e);
  double s = p + e;                        // fast two-sum (|p| >= |e|)
  return {s, e - (s - p)};
}

// mant * 10^e10, mant != 0, `inexact` when digits were dropped
__device__ __noinline__ double scale_pow10_slow(uint64_t mant, int e10) {
  if (e10 > PP_P10_MAX) return __longlong_as_double(0x7FF0000000000000ll);  // +inf
  if (e10 < PP_P10_MIN) return 0.0;
  const int k = e10 - PP_P10_MIN;
  DD p = {__ldg(&pp_p10_hi[k]), __ldg(&pp_p10_lo[k])};
  const int e2 = __ldg(&pp_p10_e2[k]);
  // mant as a double-double: hi = RN(mant), lo = mant - hi (exact, |lo| < 2^11)
  double mh = double(mant);
  double ml = double(int64_t(mant - uint64_t(mh)));
  DD r = dd_mul({mh, ml}, p);
  // r in [1, 2^65) * 2^e2; round once to binary64 and scale
  double v = r.hi + r.lo;
  return scalbn(v, e2);
}

struct FloatAcc {
  uint64_t mant = 0;
  int32_t d10 = 0;     // decimal exponent adjustment from digit positions
  int32_t ex = 0;      // explicit exponent magnitude (saturating)
  uint16_t nsig = 0;   // digits accumulated into mant
  uint16_t ndig = 0;   // digits in int + frac parts
  uint8_t phase = 0;   // 0 start, 1 int, 2 frac, 3 'e' seen, 4 exp sign, 5 exp digits, 6 error
  bool neg = false, eneg = false, inexact = false;

  __device__ __forceinline__ void digit(uint32_t d, bool frac) {
    ++ndig;
    if (nsig == 0 && d == 0) { if (frac) --d10; return; }
    if (nsig < 19) { mant = mant * 10 + d; ++nsig; if (frac) --d10; return; }
    if (!frac) ++d10;
    if (d) inexact = true;
  }
  __device__ __forceinline__ void feed(uint32_t c) {
    const uint32_t d = c - '0';
    switch (phase) {
      case 0:
        if (c == '+' || c == '-') { neg = c == '-'; phase = 1; }
        else if (d <= 9) { phase = 1; digit(d, false); }
        else if (c == '.') phase = 2;
        else phase = 6;
        break;
      case 1:
        if (d <= 9) digit(d, false);
        else if (c == '.') phase = 2;
        else if ((c | 0x20) == 'e') phase = 3;
        else phase = 6;
        break;
      case 2:
        if (d <= 9) digit(d, true);
        else if ((c | 0x20) == 'e') phase = 3;
        else phase = 6;
        break;
      case 3:
        if (c == '+' || c == '-') { eneg = c == '-'; phase = 4; }
        else if (d <= 9) { phase = 5; ex = int32_t(d); }
        else phase = 6;
        break;
      case 4:
        if (d <= 9) { phase = 5; ex = int32_t(d); } else phase = 6;
        break;
      case 5:
        if (d <= 9) ex = ex > 100000 ? ex : ex * 10 + int32_t(d);
        else phase = 6;
        break;
      default:
        break;
    }
  }
  // returns 0 or PP_ERR_NUM_SYNTAX; *out gets the value (0 on error)
  __device__ __forceinline__ int finish(double* out) const {
    *out = 0.0;
    if (phase == 6 || phase == 3 || phase == 4 || ndig == 0) return PP_ERR_NUM_SYNTAX;
    double v;
    if (mant == 0) {
      v = 0.0;
    } else {
      const int e10 = d10 + (eneg ? -ex : ex);
      if (!inexact && mant <= (1ull << 53) && e10 >= -22 && e10 <= 22) {
        const double m = double(mant);  // exact
        v = e10 >= 0 ? m * exact_pow10(e10) : m / exact_pow10(-e10);
      } else {
        v = scale_pow10_slow(mant, e10);
      }
    }
    *out = neg ? -v : v;
    return 0;
  }
};

struct IntAcc {
  uint64_t mag = 0;
  uint8_t phase = 0;  // 0 start, 1 after sign, 2 digits, 3 error
  bool neg = false, ovf = false;

  __device__ __forceinline__ void feed(uint32_t c) {
    if (phase == 0 && (c == '+' || c == '-')) { neg = c == '-'; phase = 1; return; }
    const uint32_t d = c - '0';
    if (d > 9 || phase == 3) { phase = 3; return; }
    phase = 2;
    if (mag > 1844674407370955161ull || (mag == 1844674407370955161ull && d > 5)) ovf = true;
    else mag = mag * 10 + d;
  }
  // lo_mag: magnitude allowed when negative, hi: when positive
  __device__ __forceinline__ int finish(uint64_t neg_max, uint64_t pos_max, int64_t* out) const {
    *out = 0;
    if (phase != 2) return PP_ERR_NUM_SYNTAX;
    if (ovf || mag > (neg ? neg_max : pos_max)) return PP_ERR_NUM_OVERFLOW;
    *out = neg ? int64_t(0) - int64_t(mag) : int64_t(mag);
    return 0;
  }
};

}  // namespace ppn
