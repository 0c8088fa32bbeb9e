// Streaming numeric conversion of one field's value bytes (ParPaRaw Section
// 3.3, "converting the symbol string to the column's type"; Section 4.3,
// "the empty string is parsed as the column's default value").
//
// Integers: grammar [+-]?[0-9]+, exact, range-checked per column type.
// Floats: grammar [+-]?([0-9]+(\.[0-9]*)?|\.[0-9]+)([eE][+-]?[0-9]+)?.
//
// The float conversion uses integer arithmetic only (GB300's FP64 rate is
// a small fraction of its integer rate).  With w the first 19 significant
// digits and q the decimal exponent, w * 10^q = w * 5^q * 2^q: the
// normalised w is multiplied by a 128-bit normalised power of five (the
// scheme of Lemire, "Number Parsing at a Gigabyte per Second", 2021), the
// top 54 bits of the exact 192-bit product give the significand and the
// rounding bit, the lower bits the sticky bit, and the binary64 bits are
// assembled directly (ties to even, subnormals, overflow to infinity).
// Powers 5^q with 0 <= q <= 55 are exact in the table, so every input with
// at most 19 digits and such a q converts exactly; for the other q the
// truncated table entry (relative error < 2^-127) can only matter within
// 2^-120 of a rounding tie, and dropped digits beyond the 19th only within
// 10^-18: the result is then at most 1 ulp from the correctly rounded one.
#pragma once
#include <cstdint>
#include "pp.h"

#if defined(__CUDACC__)
#define PP_FN __device__ __forceinline__
#define PP_MFN __device__ __forceinline__
#define PP_TABLE_QUAL __device__ const
#define PP_LDG(p) __ldg(p)
#else
#define PP_FN static inline
#define PP_MFN inline
#define PP_TABLE_QUAL static const
#define PP_LDG(p) (*(p))
#endif

#include "pow5_table.inc"

namespace ppn {

PP_FN void mul64x64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
#if defined(__CUDA_ARCH__)
  *hi = __umul64hi(a, b);
  *lo = a * b;
#else
  const unsigned __int128 p = (unsigned __int128)a * b;
  *hi = (uint64_t)(p >> 64);
  *lo = (uint64_t)p;
#endif
}

PP_FN int clz64(uint64_t x) {
#if defined(__CUDA_ARCH__)
  return __clzll((long long)x);
#else
  return __builtin_clzll(x);
#endif
}

// Bits of the binary64 nearest to w * 10^q (w > 0), see the file comment.
PP_FN uint64_t decimal_to_binary64(uint64_t w, int q) {
  if (q > PP_P5_MAX) return 0x7FF0000000000000ull;  // >= 10^309
  if (q < PP_P5_MIN) return 0;                      // < 2^-1075
  const int k = q - PP_P5_MIN;
  const uint64_t th = PP_LDG(&pp_p5_hi[k]);
  const uint64_t tl = PP_LDG(&pp_p5_lo[k]);
  const int e5 = PP_LDG(&pp_p5_e2[k]);
  const int lz = clz64(w);
  const uint64_t W = w << lz;
  // P = W * (th:tl) = p2:p1:p0
  uint64_t ah, al, bh, bl;
  mul64x64(W, tl, &ah, &al);
  mul64x64(W, th, &bh, &bl);
  const uint64_t p0 = al;
  uint64_t p1 = bl + ah;
  const uint64_t p2 = bh + (p1 < bl ? 1u : 0u);
  // w*10^q = P * 2^(q + e5 - 127 - lz) = p2 * 2^(1 + q + e5 - lz) + lower
  const int ub = int(p2 >> 63);             // MSB of p2 at bit 63 (1) or 62 (0)
  const int drop = 9 + ub;                  // bits of p2 below the 54 kept
  const int scale = 1 + q + e5 - lz;        // value = p2 * 2^scale
  // binary exponent of the 53-bit significand m53 (value = m53 * 2^e)
  int e = scale + drop + 1;
  const int biased = e + 1075;              // IEEE exponent field if normal
  int shift = drop + 1;                     // bits of p2 below the significand
  if (biased <= 0) {                        // subnormal: drop more bits
    shift += 1 - biased;
    if (shift > 64) return 0;               // below half the least subnormal
  }
  // m54 = significand plus one rounding bit; sticky = anything below it
  uint64_t m54, below;
  if (shift == 64) {
    m54 = p2 >> 63;
    below = p2 & ~(1ull << 63);
  } else {
    m54 = p2 >> (shift - 1);
    below = p2 & ((1ull << (shift - 1)) - 1);
  }
  const bool sticky = below != 0 || p1 != 0 || p0 != 0;
  uint64_t m = m54 >> 1;
  if ((m54 & 1) && (sticky || (m & 1))) ++m;  // round to nearest, ties to even
  if (biased <= 0) return m;                   // subnormal (m may reach 2^52: fine)
  if (m == (1ull << 53)) { m >>= 1; ++e; }
  const int be = e + 1075;
  if (be >= 2047) return 0x7FF0000000000000ull;
  return (uint64_t(be) << 52) | (m & ((1ull << 52) - 1));
}

// Bits of the binary64 nearest to w * 10^q for a short significand:
// 0 < w < 2^32 and -22 <= q <= 0 (a plain decimal such as "463.86"), with
// q == 0 the exact integer conversion.  w times the 128-bit table entry,
// truncated to its top 96 bits, carries a relative error below 2^-94; the
// value w / 10^-q is a rational whose distance from any rounding tie is
// at least 2^-86 relative (its numerator against a 54-bit dyadic differs
// by a nonzero integer), so the top 54 bits round correctly.
PP_FN uint64_t short_decimal_to_binary64(uint32_t w, int q) {
  const int lzw = clz64(uint64_t(w)) - 32;  // w != 0
  if (q == 0)
    return (uint64_t(1054 - lzw) << 52) | ((uint64_t(w) << (lzw + 21)) & ((1ull << 52) - 1));
  const int k = q - PP_P5_MIN;
  const uint64_t th = PP_LDG(&pp_p5_hi[k]);
  const uint64_t tl = PP_LDG(&pp_p5_lo[k]);
  const int e5 = PP_LDG(&pp_p5_e2[k]);
  // (w * (th:tl)) >> 64 = hi * 2^32 + lo32, with hi >= 2^31
  const uint64_t c1 = uint64_t(w) * uint32_t(tl);
  const uint64_t c2 = uint64_t(w) * uint32_t(tl >> 32) + (c1 >> 32);
  const uint64_t plo = uint64_t(w) * uint32_t(th) + (c2 >> 32);
  const uint64_t hi = uint64_t(w) * uint32_t(th >> 32) + (plo >> 32);
  const uint32_t lo32 = uint32_t(plo);
  const int L = clz64(hi);                   // 0..32
  const uint64_t top = L ? ((hi << L) | (uint64_t(lo32) >> (32 - L))) : hi;  // in [2^63, 2^64)
  // w * 10^q ~= (hi * 2^32 + lo32) * 2^(q + e5 - 63) = top * 2^(32 - L + q + e5 - 63)
  uint64_t m = (top >> 11) + ((top >> 10) & 1u);
  int be = 32 - L + q + e5 - 63 + 11 + 52 + 1023;
  if (m == (1ull << 53)) { m >>= 1; ++be; }
  return (uint64_t(be) << 52) | (m & ((1ull << 52) - 1));
}

struct FloatAcc {
  uint64_t mant = 0;
  int32_t d10 = 0;     // decimal exponent adjustment from digit positions
  int32_t ex = 0;      // explicit exponent magnitude (saturating)
  uint16_t nsig = 0;   // digits accumulated into mant
  uint16_t ndig = 0;   // digits in int + frac parts
  uint8_t phase = 0;   // 0 start, 1 int, 2 frac, 3 'e' seen, 4 exp sign, 5 exp digits, 6 error
  bool neg = false, eneg = false;

  PP_MFN void digit(uint32_t d, bool frac) {
    ++ndig;
    if (nsig == 0 && d == 0) { if (frac) --d10; return; }
    if (nsig < 19) { mant = mant * 10 + d; ++nsig; if (frac) --d10; return; }
    if (!frac) ++d10;
  }
  PP_MFN void feed(uint32_t c) {
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
  // returns 0 or PP_ERR_NUM_SYNTAX; *bits gets the binary64 bits (0 on error)
  PP_MFN int finish(uint64_t* bits) const {
    *bits = 0;
    if (phase == 6 || phase == 3 || phase == 4 || ndig == 0) return PP_ERR_NUM_SYNTAX;
    const uint64_t mag = mant == 0 ? 0 : decimal_to_binary64(mant, d10 + (eneg ? -ex : ex));
    *bits = mag | (neg ? (1ull << 63) : 0);
    return 0;
  }
};

struct IntAcc {
  uint64_t mag = 0;
  uint8_t phase = 0;  // 0 start, 1 after sign, 2 digits, 3 error
  bool neg = false, ovf = false;

  PP_MFN void feed(uint32_t c) {
    if (phase == 0 && (c == '+' || c == '-')) { neg = c == '-'; phase = 1; return; }
    const uint32_t d = c - '0';
    if (d > 9 || phase == 3) { phase = 3; return; }
    phase = 2;
    if (mag > 1844674407370955161ull || (mag == 1844674407370955161ull && d > 5)) ovf = true;
    else mag = mag * 10 + d;
  }
  // neg_max: magnitude allowed when negative, pos_max: when positive
  PP_MFN int finish(uint64_t neg_max, uint64_t pos_max, int64_t* out) const {
    *out = 0;
    if (phase != 2) return PP_ERR_NUM_SYNTAX;
    if (ovf || mag > (neg ? neg_max : pos_max)) return PP_ERR_NUM_OVERFLOW;
    *out = neg ? int64_t(~mag + 1) : int64_t(mag);
    return 0;
  }
};

}  // namespace ppn
