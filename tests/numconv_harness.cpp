// Host build of the library's numeric field conversion (pp_numeric.cuh) so
// that its arithmetic can be checked on the CPU against an independent,
// correctly rounded conversion.  Not part of the library.
#include <cstddef>
#include <cstdint>
#include "pp_numeric.cuh"

extern "C" {
// `buf` holds n strings, each terminated by one 0x00 byte.  For each:
// bits[i] = binary64 bits, err[i] = 0 / PP_ERR_NUM_SYNTAX.
void h_parse_floats(const unsigned char* buf, size_t n, uint64_t* bits, int* err) {
  size_t p = 0;
  for (size_t i = 0; i < n; ++i) {
    ppn::FloatAcc a;
    while (buf[p]) a.feed(buf[p++]);
    ++p;
    err[i] = a.finish(&bits[i]);
  }
}
uint64_t h_decimal_to_binary64(uint64_t w, int q) { return ppn::decimal_to_binary64(w, q); }
uint64_t h_short_decimal_to_binary64(uint32_t w, int q) {
  return ppn::short_decimal_to_binary64(w, -q);
}
// the 8 bytes at s as a short plain decimal of n characters
int h_short_decimal(const unsigned char* s, int n, int dot, uint32_t* w, int* k) {
  uint32_t x0 = 0, x1 = 0;
  for (int i = 0; i < 4; ++i) x0 |= uint32_t(s[i]) << (8 * i);
  for (int i = 0; i < 4; ++i) x1 |= uint32_t(s[4 + i]) << (8 * i);
  return ppn::short_decimal(x0, x1, n, dot != 0, w, k) ? 1 : 0;
}
}

extern "C" {
// `buf` holds n fields, each terminated by one 0x00 byte, as timestamps:
// out[i] = seconds since 1970, err[i] = 0 / PP_ERR_NUM_SYNTAX.
void h_parse_timestamps(const unsigned char* buf, size_t n, int64_t* out, int* err) {
  size_t p = 0;
  for (size_t i = 0; i < n; ++i) {
    ppn::TsAcc a;
    while (buf[p]) a.feed(buf[p++]);
    ++p;
    err[i] = a.finish(&out[i]);
  }
}
int64_t h_days_from_civil(int y, int m, int d) { return ppn::days_from_civil(y, m, d); }
}
