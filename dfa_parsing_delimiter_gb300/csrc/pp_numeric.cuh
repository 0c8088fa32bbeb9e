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

PP_FN int clz32(uint32_t x) {
#if defined(__CUDA_ARCH__)
  return __clz(int(x));
#else
  return x ? __builtin_clz(x) : 32;
#endif
}
PP_FN int ctz32(uint32_t x) {  // x != 0
#if defined(__CUDA_ARCH__)
  return __ffs(int(x)) - 1;
#else
  return __builtin_ctz(x);
#endif
}
PP_FN int popc32(uint32_t x) {
#if defined(__CUDA_ARCH__)
  return __popc(x);
#else
  return __builtin_popcount(x);
#endif
}
PP_FN uint32_t umulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return uint32_t((uint64_t(a) * b) >> 32);
#endif
}
// Byte permute with PTX prmt semantics (default mode): result byte i is
// byte (s >> 4i) & 7 of the eight bytes b:a (a the low word); when bit 3 of
// that nibble is set, the chosen byte's sign bit is replicated instead.
PP_FN uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t s) {
#if defined(__CUDA_ARCH__)
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(s));
  return r;
#else
  const uint64_t v = (uint64_t(b) << 32) | a;
  uint32_t r = 0;
  for (int i = 0; i < 4; ++i) {
    const uint32_t n = (s >> (4 * i)) & 0xFu;
    uint32_t x = uint32_t(v >> (8 * (n & 7u))) & 0xFFu;
    if (n & 8u) x = (x & 0x80u) ? 0xFFu : 0u;
    r |= x << (8 * i);
  }
  return r;
#endif
}

// ------------------------------------------------ short plain decimals
// Word-parallel decoding of a field of at most 8 characters, four to a
// 32-bit word (character i in byte i).  With y = chars ^ '0', digits map
// to 0..9 and '.' to 0x1E.

// 0x80 in each byte of y that is not a digit
PP_FN uint32_t nondigit_bytes(uint32_t y) {
  return (((y & 0x7F7F7F7Fu) + 0x76767676u) | y) & 0x80808080u;
}
// value of the four digits in w, byte 0 the most significant
PP_FN uint32_t val4(uint32_t w) {
  w = (w * 10u + (w >> 8)) & 0x00FF00FFu;
  return (w * 100u + (w >> 16)) & 0xFFFFu;
}

// The n (1..8) characters in x0:x1 as a plain decimal: digits only, or
// (dot) digits with one '.' and at least one digit ("12", "4.5", "7.",
// ".25").  Bytes past the n-th are ignored.  On success *w = the digits
// as an integer (< 10^8) and *k = the number of digits after the '.', so
// the value is w * 10^-k.
PP_FN bool short_decimal(uint32_t x0, uint32_t x1, int n, bool dot, uint32_t* w, int* k) {
  const uint32_t y0 = x0 ^ 0x30303030u, y1 = x1 ^ 0x30303030u;
  const uint32_t m0 = n >= 4 ? 0x80808080u : 0x80808080u >> (32 - 8 * n);
  const uint32_t m1 = n <= 4 ? 0u : 0x80808080u >> (64 - 8 * n);
  const uint32_t d0 = nondigit_bytes(y0) & m0, d1 = nondigit_bytes(y1) & m1;
  int p = 8, nd = n;  // position of the '.' (8: none), digit count
  if (d0 | d1) {
    const int b = d0 ? (ctz32(d0) >> 3) : 4 + (ctz32(d1) >> 3);
    const uint32_t yb = ((b < 4 ? y0 : y1) >> (8 * (b & 3))) & 0xFFu;
    if (!dot || popc32(d0) + popc32(d1) != 1 || yb != 0x1Eu || n == 1) return false;
    p = b;
    nd = n - 1;
  }
  // Right-align the digits, dropping the '.': byte i of z0:z1 takes digit
  // i - a (a = 8 - nd leading zero bytes), i.e. character i - a, or
  // i - a + 1 from the '.' on.  The leading bytes use selector 8, the sign
  // of character 0, which is 0 for a digit or '.'.
  const int a = 8 - nd;
  uint32_t sel = (0x76543210u << (4 * a)) | (0x88888888u & ((1u << (4 * a)) - 1u));
  if (a + p < 8) sel += 0x11111111u << (4 * (a + p));
  const uint32_t z0 = byte_perm(y0, y1, sel), z1 = byte_perm(y0, y1, sel >> 16);
  *w = val4(z0) * 10000u + val4(z1);
  *k = p < 8 ? nd - p : 0;
  return true;
}

// Bits of the binary64 nearest to w * 10^-k for 0 < w < 2^32 and
// 0 <= k <= PP_R10_MAX (a plain decimal such as "463.86": w = 46386,
// k = 2).  With W = w normalised to [2^31, 2^32) and R = the table's
// 96-bit reciprocal ceil(2^(95 + e) / 10^k) (e = ceil(log2 10^k)), the top
// 64 bits T of W * R are computed exactly with three 32x32 products; the
// binary64 significand is T rounded to 53 bits.  Rounding R up keeps the
// product at or above the exact value, by less than 2^-41 units of the
// 54th bit; the exact value, a rational with denominator 5^k, is either
// dyadic (and then ends in zeros there) or at least 5^-k >= 2^-40 such
// units from a rounding point, so the rounding is always correct, and a
// tie cannot occur (it would need 54 significant bits, w has at most 32).
PP_FN uint64_t short_decimal_to_binary64(uint32_t w, int k) {
  const int lz = clz32(w);
  const uint32_t W = w << lz;
#if defined(__CUDA_ARCH__)
  const uint4 r = __ldg(reinterpret_cast<const uint4*>(pp_r10) + k);
  const uint32_t r0 = r.x, r1 = r.y, r2 = r.z;
  const int e = int(r.w);
#else
  const uint32_t r0 = pp_r10[4 * k], r1 = pp_r10[4 * k + 1], r2 = pp_r10[4 * k + 2];
  const int e = int(pp_r10[4 * k + 3]);
#endif
  const uint64_t m1 = uint64_t(W) * r1 + umulhi32(W, r0);
  const uint64_t T = uint64_t(W) * r2 + (m1 >> 32);  // in [2^62, 2^64)
  const int h = int(T >> 63);
  const uint64_t m = ((T >> (9 + h)) + 1u) >> 1;     // 53 bits (2^53 after a carry)
  // value = m * 2^(E - 52) with E = 31 + h - lz - e; adding m carries its
  // leading bit into the exponent field
  return (uint64_t(31 + h - lz - e + 1022) << 52) + m;
}

struct FloatAcc {
  uint64_t mant = 0;
  int32_t d10 = 0;     // decimal exponent adjustment from digit positions
  int32_t ex = 0;      // explicit exponent magnitude (saturating)
  uint16_t nsig = 0;   // digits accumulated into mant
  bool dig = false;    // a digit of the int or frac part seen
  uint8_t phase = 0;   // 0 start, 1 int, 2 frac, 3 'e' seen, 4 exp sign, 5 exp digits, 6 error
  bool neg = false, eneg = false;

  PP_MFN void digit(uint32_t d, bool frac) {
    dig = true;
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
    if (phase == 6 || phase == 3 || phase == 4 || !dig) return PP_ERR_NUM_SYNTAX;
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

// ------------------------------------------------------------ timestamps
// Temporal fields (ParPaRaw Section 3.3, "numerical or temporal types"):
// YYYY-MM-DD or YYYY-MM-DD HH:MM:SS (n = 10 or 19 characters) as int64
// seconds since 1970-01-01 00:00:00, proleptic Gregorian calendar, no time
// zone; month 01-12, day within the month, hour 00-23, minute and second
// 00-59.  The characters come as five little-endian words x[0..4] (byte i
// of the field in byte i % 4 of x[i / 4]; bytes past n are ignored).

// Days from 1970-01-01 to y-m-d, by the closed form of H. Hinnant's
// "chrono-Compatible Low-Level Date Algorithms" (days_from_civil): counting
// years from March makes the leap day the last day of a year, so the day of
// that year is (153 * month + 2) / 5 + day - 1 with March as month 0, and a
// 400-year era holds 146097 days; 719468 is the day of 1970-01-01 counted
// from 0000-03-01.
PP_FN int64_t days_from_civil(int y, int m, int d) {
  y -= m <= 2 ? 1 : 0;
  const int era = (y >= 0 ? y : y - 399) / 400;
  const int yoe = y - era * 400;                          // year of the era, 0..399
  const int doy = (153 * (m > 2 ? m - 3 : m + 9) + 2) / 5 + d - 1;
  const int doe = yoe * 365 + yoe / 4 - yoe / 100 + doy;  // day of the era
  return int64_t(era) * 146097 + doe - 719468;
}

// digit pair at bytes i, i+1 of y (a field word xor '0' in every byte)
PP_FN int digit_pair(uint32_t y, int i) {
  return int((y >> (8 * i)) & 0xFFu) * 10 + int((y >> (8 * i + 8)) & 0xFFu);
}

PP_FN int parse_timestamp(const uint32_t (&x)[5], uint32_t n, int64_t* out) {
  *out = 0;
  if (n == 0) return 0;
  if (n != 10 && n != 19) return PP_ERR_NUM_SYNTAX;
  const uint32_t Z = 0x30303030u;
  const uint32_t y0 = x[0] ^ Z, y1 = x[1] ^ Z, y2 = x[2] ^ Z, y3 = x[3] ^ Z, y4 = x[4] ^ Z;
  // digits where the grammar puts them, separators in between
  uint32_t bad = nondigit_bytes(y0) | (nondigit_bytes(y1) & 0x00808000u);
  bool sep = (x[1] & 0xFF0000FFu) == 0x2D00002Du;  // '-' . . '-'
  if (n == 19) {
    bad |= (nondigit_bytes(y2) & 0x80008080u) | (nondigit_bytes(y3) & 0x80800080u) |
            (nondigit_bytes(y4) & 0x00808000u);
    sep = sep && (x[2] & 0x00FF0000u) == 0x00200000u && (x[3] & 0x0000FF00u) == 0x00003A00u &&
          (x[4] & 0xFFu) == 0x3Au;  // ' ', ':', ':'
  } else {
    bad |= nondigit_bytes(y2) & 0x00008080u;
  }
  if (bad || !sep) return PP_ERR_NUM_SYNTAX;
  const int yr = int(val4(y0)), mo = digit_pair(y1, 1), d = digit_pair(y2, 0);
  int h = 0, mi = 0, sc = 0;
  if (n == 19) {
    h = int((y2 >> 24) & 0xFFu) * 10 + int(y3 & 0xFFu);
    mi = digit_pair(y3, 2);
    sc = digit_pair(y4, 1);
  }
  const bool leap = (yr % 4 == 0 && yr % 100 != 0) || yr % 400 == 0;
  // days in month m: 30 + (m + m / 8) % 2 for m != 2
  const int dim = mo == 2 ? (leap ? 29 : 28) : 30 + ((mo + mo / 8) & 1);
  if (mo < 1 || mo > 12 || d < 1 || d > dim || h > 23 || mi > 59 || sc > 59)
    return PP_ERR_NUM_SYNTAX;
  *out = days_from_civil(yr, mo, d) * 86400 + int64_t(h * 3600 + mi * 60 + sc);
  return 0;
}

// The same over a field fed byte by byte (fields that are not plain bytes
// of the current tile).
struct TsAcc {
  uint32_t x[5] = {0u, 0u, 0u, 0u, 0u};
  uint32_t n = 0;
  PP_MFN void feed(uint32_t c) {
    if (n < 20) x[n >> 2] |= (c & 0xFFu) << (8 * (n & 3));
    ++n;
  }
  PP_MFN int finish(int64_t* out) const { return parse_timestamp(x, n, out); }
};

}  // namespace ppn
