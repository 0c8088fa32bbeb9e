/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow, single-threaded CPU statement of what the parser computes,
 * used to check the GPU library.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header or table with the CUDA library.
 *
 * Source: "ParPaRaw: Massively Parallel Parsing of Delimiter-Separated Raw
 * Data" (Sections 3.1-3.4 and 4, Figures 2-5).  The method is only a fast
 * route to the result of sequential DFA parsing (Section 3.1: "A sequential
 * approach would simply set the starting state of its DFA and read the
 * symbols of the input beginning to end"), so the oracle *is* that
 * sequential walk:
 *   - walk the DFA from the start state byte by byte,
 *   - classify each byte from (state before, symbol),
 *   - append value bytes to the current field,
 *   - close the field at every field/record delimiter, close the record at
 *     every record delimiter.
 * The DFA tables are written as switch statements from the state names
 * EOR/FLD/ENC/ESC/INV (Section 3.1, Figure 3 and its caption about the
 * invalid state, "reading quotes in FLD state").
 *
 * The method's own steps (multi-instance DFA -> state-transition vector,
 * composite operation, exclusive scan; absolute/relative column offsets;
 * the per-chunk column-count aggregate) are stated separately below
 * (or_stv_*, or_colofs_*, or_fields_*) so the tests can check them against
 * the sequential walk on every short input.
 *
 * Also stated plainly: timestamps (conv_ts: days counted a year and a month
 * at a time), CRLF line ends (a CR symbol, kind 2), the fewest and most
 * fields per record (or_count_fields), and symbols of several bytes in
 * UTF-8 and UTF-16 inputs (sym_at, or_csv_parse_enc: the DFA steps once per
 * symbol, decoded front to back).
 *
 * The JSON-like lexer DFA (16 states) follows the prefix-scan lexing scheme
 * of "Lexing on the GPU: the scan is the easy part" (section "A lexer is a
 * prefix scan"): one transition function per input symbol; a token begins
 * where the automaton leaves a finished token for a new one.
 *
 * Floats: glibc strtod (correctly rounded, round-half-even).
 */
#include <errno.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ codes */
/* error bits (a bitmask); the same values are part of the library's ABI   */
#define E_INVALID_INPUT 1
#define E_BAD_END_STATE 2
#define E_COLCOUNT 4
#define E_NUM_SYNTAX 8
#define E_NUM_OVERFLOW 16
#define E_CAPACITY 32

enum { T_DATA = 0, T_FD = 1, T_RD = 2, T_CTRL = 3, T_INVALID = 4, T_BEGIN = 5 };
enum { C_STR = 0, C_I8 = 1, C_I32 = 2, C_I64 = 3, C_F64 = 4, C_SKIP = 5, C_TS = 6 };

typedef struct {
  int32_t error;
  int32_t pad;
  uint64_t first_error_offset;
  uint64_t n_records;
  uint64_t n_tokens;
  uint64_t chars_len[64];
  uint64_t n_dropped;          /* records not emitted (skipped or rejected) */
} or_status;

static void flag(or_status* st, int bit, uint64_t off, int with_offset) {
  st->error |= bit;
  if (with_offset && off < st->first_error_offset) st->first_error_offset = off;
}

/* ------------------------------------------------------------ CSV DFA */
enum { EOR = 0, FLD = 1, ENC = 2, ESC = 3, INV = 4 };

/* The symbols the CSV DFA tells apart, as byte values or, for the
 * encodings below, code points; cr: a carriage return dropped outside
 * quotes (CRLF line ends), or -1 */
typedef struct { uint32_t fd, rd, q; int64_t cr; } csv_syms;

/* One transition of the quoted-CSV DFA.  Returns the next state and writes
 * the symbol's tag.  Cells (state, symbol) -> (next, tag):
 *   EOR: quote -> ENC ctrl | fd -> EOR fd | rd -> EOR rd | other -> FLD data
 *   FLD: quote -> INV      | fd -> EOR fd | rd -> EOR rd | other -> FLD data
 *   ENC: quote -> ESC ctrl | anything else -> ENC data
 *   ESC: quote -> ENC data (second quote of a doubled pair)
 *        fd -> EOR fd | rd -> EOR rd | other -> INV
 *   INV: everything -> INV
 * With a carriage return byte (CRLF line ends: the pages name no line-end
 * convention, and ParPaRaw Section 4 notes that simulating the DFA allows
 * more expressive parsing rules), a CR outside quotes is a control symbol,
 * dropped from the value, that leaves the field open:
 *   EOR, FLD, ESC: cr -> FLD ctrl     ENC: cr -> ENC data                */
static int csv_step(const csv_syms* y, int s, uint32_t b, int* tag) {
  int is_q = b == y->q, is_fd = b == y->fd, is_rd = b == y->rd, is_cr = (int64_t)b == y->cr;
  switch (s) {
    case EOR:
      if (is_q) { *tag = T_CTRL; return ENC; }
      if (is_fd) { *tag = T_FD; return EOR; }
      if (is_rd) { *tag = T_RD; return EOR; }
      if (is_cr) { *tag = T_CTRL; return FLD; }
      *tag = T_DATA; return FLD;
    case FLD:
      if (is_q) { *tag = T_INVALID; return INV; }
      if (is_fd) { *tag = T_FD; return EOR; }
      if (is_rd) { *tag = T_RD; return EOR; }
      if (is_cr) { *tag = T_CTRL; return FLD; }
      *tag = T_DATA; return FLD;
    case ENC:
      if (is_q) { *tag = T_CTRL; return ESC; }
      *tag = T_DATA; return ENC;
    case ESC:
      if (is_q) { *tag = T_DATA; return ENC; }
      if (is_fd) { *tag = T_FD; return EOR; }
      if (is_rd) { *tag = T_RD; return EOR; }
      if (is_cr) { *tag = T_CTRL; return FLD; }
      *tag = T_INVALID; return INV;
    default:
      *tag = T_INVALID; return INV;
  }
}
static int csv_accepting(int s) { return s == EOR || s == FLD || s == ESC; }

/* ------------------------------------------------------------ lexer DFA */
enum { L_START = 0, L_WS, L_PUNCT, L_STR_OPEN, L_STR, L_STR_BSL, L_STR_END, L_NEG,
       L_ZERO, L_INT, L_DOT, L_FRAC, L_EXP_E, L_EXP_SIGN, L_EXP, L_INV };
enum { G_WS = 0, G_PUNCT, G_QUOTE, G_BSL, G_MINUS, G_PLUS, G_ZERO, G_D19, G_DOT,
       G_E, G_OTHER };

static int lex_group(uint8_t b) {
  switch (b) {
    case ' ': case '\t': case '\n': case '\r': return G_WS;
    case '{': case '}': case '[': case ']': case ',': case ':': return G_PUNCT;
    case '"': return G_QUOTE;
    case '\\': return G_BSL;
    case '-': return G_MINUS;
    case '+': return G_PLUS;
    case '0': return G_ZERO;
    case '.': return G_DOT;
    case 'e': case 'E': return G_E;
    default: return (b >= '1' && b <= '9') ? G_D19 : G_OTHER;
  }
}
/* the state that starts a new token on symbol group g (INV if none) */
static int lex_begin(int g) {
  switch (g) {
    case G_WS: return L_WS;
    case G_PUNCT: return L_PUNCT;
    case G_QUOTE: return L_STR_OPEN;
    case G_MINUS: return L_NEG;
    case G_ZERO: return L_ZERO;
    case G_D19: return L_INT;
    default: return L_INV;
  }
}
static int ends_number(int g) { return g == G_WS || g == G_PUNCT || g == G_QUOTE || g == G_MINUS; }

/* One lexer transition; *begin = 1 when a new token starts at this byte. */
static int lex_step(int s, uint8_t b, int* begin) {
  int g = lex_group(b), n;
  *begin = 0;
  switch (s) {
    case L_START: case L_WS: case L_PUNCT: case L_STR_END:
      n = lex_begin(g);
      *begin = (n != L_INV) && !(s == L_WS && g == G_WS);
      return n;
    case L_STR_OPEN: case L_STR:
      return g == G_QUOTE ? L_STR_END : g == G_BSL ? L_STR_BSL : L_STR;
    case L_STR_BSL:
      return L_STR;
    case L_NEG:
      return g == G_ZERO ? L_ZERO : g == G_D19 ? L_INT : L_INV;
    case L_ZERO:
      if (g == G_DOT) return L_DOT;
      if (g == G_E) return L_EXP_E;
      if (ends_number(g)) { *begin = 1; return lex_begin(g); }
      return L_INV;
    case L_INT:
      if (g == G_ZERO || g == G_D19) return L_INT;
      if (g == G_DOT) return L_DOT;
      if (g == G_E) return L_EXP_E;
      if (ends_number(g)) { *begin = 1; return lex_begin(g); }
      return L_INV;
    case L_DOT:
      return (g == G_ZERO || g == G_D19) ? L_FRAC : L_INV;
    case L_FRAC:
      if (g == G_ZERO || g == G_D19) return L_FRAC;
      if (g == G_E) return L_EXP_E;
      if (ends_number(g)) { *begin = 1; return lex_begin(g); }
      return L_INV;
    case L_EXP_E:
      if (g == G_PLUS || g == G_MINUS) return L_EXP_SIGN;
      return (g == G_ZERO || g == G_D19) ? L_EXP : L_INV;
    case L_EXP_SIGN:
      return (g == G_ZERO || g == G_D19) ? L_EXP : L_INV;
    case L_EXP:
      if (g == G_ZERO || g == G_D19) return L_EXP;
      if (ends_number(g)) { *begin = 1; return lex_begin(g); }
      return L_INV;
    default:
      return L_INV;
  }
}
static int lex_accepting(int s) {
  return s == L_START || s == L_WS || s == L_PUNCT || s == L_STR_END || s == L_ZERO ||
         s == L_INT || s == L_FRAC || s == L_EXP;
}
/* token id from the state after the token's last byte */
static int lex_token_id(int s, uint8_t first_byte) {
  switch (s) {
    case L_WS: return 9;
    case L_PUNCT:
      switch (first_byte) {
        case '{': return 0; case '}': return 1; case '[': return 2;
        case ']': return 3; case ',': return 4; default: return 5;
      }
    case L_STR_END: return 6;
    case L_ZERO: case L_INT: return 7;
    case L_FRAC: case L_EXP: return 8;
    default: return 255;
  }
}

/* ------------------------------------------------- generic step by kind */
/* kind 0 = quoted CSV (syms from y), kind 1 = JSON-like lexer, kind 2 =
 * quoted CSV with CRLF line ends (CR dropped outside quotes)               */
static int is_csv(int kind) { return kind == 0 || kind == 2; }
static csv_syms syms_of(int kind, uint8_t fd, uint8_t rd, uint8_t q) {
  csv_syms y = {fd, rd, q, kind == 2 ? '\r' : -1};
  return y;
}
static int step_any(int kind, const csv_syms* y, int s, uint8_t b, int* tag) {
  if (is_csv(kind)) return csv_step(y, s, b, tag);
  int begin, n = lex_step(s, b, &begin);
  *tag = n == L_INV ? T_INVALID : begin ? T_BEGIN : T_DATA;
  return n;
}
static int nstates(int kind) { return is_csv(kind) ? 5 : 16; }

/* Per-byte state before and tag (the test hook's definition). */
int or_tags(int kind, uint8_t fd, uint8_t rd, uint8_t q, const uint8_t* in, uint64_t n,
            uint8_t* state_before, uint8_t* tag) {
  csv_syms y = syms_of(kind, fd, rd, q);
  int s = is_csv(kind) ? EOR : L_START;
  for (uint64_t i = 0; i < n; i++) {
    int t;
    state_before[i] = (uint8_t)s;
    s = step_any(kind, &y, s, in[i], &t);
    tag[i] = (uint8_t)t;
  }
  return s;
}

/* ------------------------------------------------------ numeric fields */
/* Integer grammar [+-]?[0-9]+ over the field's value bytes.  Returns 0 ok,
 * E_NUM_SYNTAX or E_NUM_OVERFLOW; the value is 0 on error and for "".     */
static int conv_int(const uint8_t* v, size_t n, int64_t lo, int64_t hi, int64_t* out) {
  *out = 0;
  if (n == 0) return 0;
  size_t i = 0;
  int neg = 0;
  if (v[0] == '+' || v[0] == '-') { neg = v[0] == '-'; i = 1; }
  if (i == n) return E_NUM_SYNTAX;
  for (size_t k = i; k < n; k++)
    if (v[k] < '0' || v[k] > '9') return E_NUM_SYNTAX;
  /* magnitude with saturation above 2^63 */
  unsigned __int128 mag = 0;
  const unsigned __int128 CAP = ((unsigned __int128)1) << 64;
  for (; i < n; i++) {
    mag = mag * 10 + (unsigned)(v[i] - '0');
    if (mag > CAP) mag = CAP;
  }
  __int128 val = neg ? -(__int128)mag : (__int128)mag;
  if (val < lo || val > hi) return E_NUM_OVERFLOW;
  *out = (int64_t)val;
  return 0;
}

/* Float grammar [+-]?([0-9]+(\.[0-9]*)?|\.[0-9]+)([eE][+-]?[0-9]+)?; the
 * value is strtod's (correctly rounded).  "" -> 0.0.                      */
static int conv_f64(const uint8_t* v, size_t n, double* out) {
  *out = 0.0;
  if (n == 0) return 0;
  size_t i = 0, d0 = 0, d1 = 0;
  if (v[i] == '+' || v[i] == '-') i++;
  while (i < n && v[i] >= '0' && v[i] <= '9') { i++; d0++; }
  if (i < n && v[i] == '.') {
    i++;
    while (i < n && v[i] >= '0' && v[i] <= '9') { i++; d1++; }
  }
  if (d0 + d1 == 0) return E_NUM_SYNTAX;
  if (i < n && (v[i] == 'e' || v[i] == 'E')) {
    i++;
    if (i < n && (v[i] == '+' || v[i] == '-')) i++;
    size_t de = 0;
    while (i < n && v[i] >= '0' && v[i] <= '9') { i++; de++; }
    if (de == 0) return E_NUM_SYNTAX;
  }
  if (i != n) return E_NUM_SYNTAX;
  char stackbuf[128];
  char* s = n < sizeof stackbuf ? stackbuf : (char*)malloc(n + 1);
  memcpy(s, v, n);
  s[n] = 0;
  *out = strtod(s, NULL);
  if (s != stackbuf) free(s);
  return 0;
}

/* Temporal fields (ParPaRaw Section 3.3, field values of "numerical or
 * temporal types"; the pages fix no format).  Reading: YYYY-MM-DD or
 * YYYY-MM-DD HH:MM:SS, four- and two-digit fields, month 01-12, day within
 * the month of the proleptic Gregorian calendar, hour 00-23, minute and
 * second 00-59; the value is the signed count of seconds since 1970-01-01
 * 00:00:00 (no time zone).  "" -> 0; anything else E_NUM_SYNTAX and 0.
 * The days are counted one year and one month at a time, the plain way. */
static int is_leap(int y) { return (y % 4 == 0 && y % 100 != 0) || y % 400 == 0; }
static int month_days(int y, int m) {
  static const int d[12] = {31, 28, 31, 30, 31, 30, 31, 31, 30, 31, 30, 31};
  return m == 2 && is_leap(y) ? 29 : d[m - 1];
}
static int two(const uint8_t* v, size_t i, int* out) {
  if (v[i] < '0' || v[i] > '9' || v[i + 1] < '0' || v[i + 1] > '9') return 0;
  *out = (v[i] - '0') * 10 + (v[i + 1] - '0');
  return 1;
}
static int conv_ts(const uint8_t* v, size_t n, int64_t* out) {
  *out = 0;
  if (n == 0) return 0;
  if (n != 10 && n != 19) return E_NUM_SYNTAX;
  int yh, yl, mo, d, h = 0, mi = 0, sec = 0;
  if (!two(v, 0, &yh) || !two(v, 2, &yl) || v[4] != '-' || !two(v, 5, &mo) || v[7] != '-' ||
      !two(v, 8, &d))
    return E_NUM_SYNTAX;
  if (n == 19 && (v[10] != ' ' || !two(v, 11, &h) || v[13] != ':' || !two(v, 14, &mi) ||
                  v[16] != ':' || !two(v, 17, &sec)))
    return E_NUM_SYNTAX;
  const int y = yh * 100 + yl;
  if (mo < 1 || mo > 12 || d < 1 || d > month_days(y, mo) || h > 23 || mi > 59 || sec > 59)
    return E_NUM_SYNTAX;
  int64_t days = 0;
  for (int k = 1970; k < y; k++) days += is_leap(k) ? 366 : 365;
  for (int k = y; k < 1970; k++) days -= is_leap(k) ? 366 : 365;
  for (int k = 1; k < mo; k++) days += month_days(y, k);
  days += d - 1;
  *out = days * 86400 + (int64_t)h * 3600 + mi * 60 + sec;
  return 0;
}

/* ------------------------------------------------------------ CSV parse */
typedef struct {
  /* outputs */
  int n_cols;
  const int32_t* types;
  const uint64_t* defaults;     /* bits stored for an empty or missing numeric field, or NULL */
  int32_t** offsets;
  uint8_t** chars;
  void** typed;
  uint64_t rec_cap;
  const uint64_t* chars_cap;
  or_status* st;
  /* current field */
  uint8_t* val;
  size_t val_len, val_cap;
} csv_out;

static void field_value_push(csv_out* o, uint8_t b) {
  if (o->val_len == o->val_cap) {
    o->val_cap = o->val_cap ? 2 * o->val_cap : 256;
    o->val = (uint8_t*)realloc(o->val, o->val_cap);
  }
  o->val[o->val_len++] = b;
}

/* Close field `col` of record `rec`; the value is o->val. */
static void close_field(csv_out* o, uint64_t rec, int col, uint64_t field_start) {
  if (col >= o->n_cols) return;                 /* extra field: dropped */
  int t = o->types[col];
  if (t == C_SKIP) return;
  if (rec >= o->rec_cap) { flag(o->st, E_CAPACITY, 0, 0); return; }
  if (t == C_STR) {
    uint64_t len = o->st->chars_len[col];
    if (len + o->val_len > o->chars_cap[col] || len + o->val_len > 0x7FFFFFFFull) {
      flag(o->st, E_CAPACITY, 0, 0);
      return;
    }
    memcpy(o->chars[col] + len, o->val, o->val_len);
    len += o->val_len;
    o->st->chars_len[col] = len;
    o->offsets[col][rec + 1] = (int32_t)len;
    return;
  }
  int rc;
  if (o->val_len == 0 && o->defaults) {       /* empty or missing: the column default */
    const uint64_t d = o->defaults[col];
    if (t == C_I8) ((int8_t*)o->typed[col])[rec] = (int8_t)d;
    else if (t == C_I32) ((int32_t*)o->typed[col])[rec] = (int32_t)d;
    else ((uint64_t*)o->typed[col])[rec] = d;
    return;
  }
  if (t == C_F64) {
    double d;
    rc = conv_f64(o->val, o->val_len, &d);
    ((double*)o->typed[col])[rec] = d;
  } else if (t == C_TS) {
    int64_t x;
    rc = conv_ts(o->val, o->val_len, &x);
    ((int64_t*)o->typed[col])[rec] = x;
  } else {
    int64_t lo = t == C_I8 ? -128 : t == C_I32 ? INT32_MIN : INT64_MIN;
    int64_t hi = t == C_I8 ? 127 : t == C_I32 ? INT32_MAX : INT64_MAX;
    int64_t x;
    rc = conv_int(o->val, o->val_len, lo, hi, &x);
    if (t == C_I8) ((int8_t*)o->typed[col])[rec] = (int8_t)x;
    else if (t == C_I32) ((int32_t*)o->typed[col])[rec] = (int32_t)x;
    else ((int64_t*)o->typed[col])[rec] = x;
  }
  if (rc) flag(o->st, rc, field_start, 1);
}

/* Close record `rec` whose last field was column `col` (terminator at off). */
static void close_record(csv_out* o, uint64_t rec, int col, uint64_t off) {
  if (col != o->n_cols - 1) flag(o->st, E_COLCOUNT, off, 1);
  o->val_len = 0;
  for (int c = col + 1; c < o->n_cols; c++) close_field(o, rec, c, off);  /* defaults */
}

/* ------------------------------------------------- symbols of an encoding */
/* ParPaRaw Section 3.4: with a variable-length encoding a symbol spans
 * several bytes; the DFA takes one transition per symbol.
 *   bytes (0): every byte is a symbol, its value the byte.
 *   UTF-8 (1): a symbol is a byte that is not a continuation byte
 *     (0b10xxxxxx) together with all the continuation bytes after it (so a
 *     chunk's leading continuation bytes belong to the symbol before).  It
 *     is well formed if it has the length its first byte announces (1 for
 *     0xxxxxxx, 2, 3, 4 for 110xxxxx, 1110xxxx, 11110xxx), is no overlong
 *     form and is at most 0x10FFFF; its value is then the code point.
 *     Continuation bytes at the input's start form one ill-formed symbol.
 *   UTF-16LE (2): 2-byte little-endian units counted from the input's first
 *     byte; a high surrogate (0xD800-0xDBFF) followed by a low surrogate
 *     (0xDC00-0xDFFF) is one 4-byte symbol, any other unit a 2-byte one
 *     whose value is the unit; an odd last byte is an ill-formed symbol.
 * sym_at returns the end of the symbol starting at i and its value in
 * *cp (OR_BAD_CP when ill formed).                                      */
#define OR_BAD_CP 0xFFFFFFFFu
static int is_cont(uint8_t b) { return (b & 0xC0) == 0x80; }
static uint64_t sym_at(const uint8_t* in, uint64_t n, int enc, uint64_t i, uint32_t* cp) {
  if (enc == 0) { *cp = in[i]; return i + 1; }
  if (enc == 1) {
    uint64_t j = i + 1;
    while (j < n && is_cont(in[j])) j++;
    const uint64_t len = j - i;
    const uint8_t b = in[i];
    uint64_t want;
    uint32_t v;
    if (b < 0x80) { want = 1; v = b; }
    else if ((b & 0xE0) == 0xC0) { want = 2; v = b & 0x1F; }
    else if ((b & 0xF0) == 0xE0) { want = 3; v = b & 0x0F; }
    else if ((b & 0xF8) == 0xF0) { want = 4; v = b & 0x07; }
    else { *cp = OR_BAD_CP; return j; }          /* a continuation byte or 0xF8-0xFF */
    if (len != want) { *cp = OR_BAD_CP; return j; }
    for (uint64_t k = i + 1; k < j; k++) v = (v << 6) | (in[k] & 0x3F);
    static const uint32_t min_of_len[5] = {0, 0, 0x80, 0x800, 0x10000};
    *cp = (v < min_of_len[len] || v > 0x10FFFF) ? OR_BAD_CP : v;
    return j;
  }
  /* UTF-16LE */
  if (i + 1 >= n) { *cp = OR_BAD_CP; return n; }
  const uint32_t u = in[i] | (uint32_t)in[i + 1] << 8;
  if (u >= 0xD800 && u <= 0xDBFF && i + 3 < n) {
    const uint32_t w = in[i + 2] | (uint32_t)in[i + 3] << 8;
    if (w >= 0xDC00 && w <= 0xDFFF) {
      *cp = 0x10000 + ((u - 0xD800) << 10) + (w - 0xDC00);
      return i + 4;
    }
  }
  *cp = u;
  return i + 2;
}

/* One parsed field of the record being collected (the records are buffered
 * whole so that a record can be dropped once its field count is known). */
typedef struct { uint64_t start, vbeg, vlen; } or_field;

static int csv_parse_core(const uint8_t* in, uint64_t n, int enc, csv_syms y,
                          int n_cols, const int32_t* col_types, const uint64_t* defaults,
                          int reject, const uint64_t* skip_records, uint64_t n_skip_records,
                          int32_t** out_offsets, uint8_t** out_chars, void** out_typed,
                          uint64_t records_capacity, const uint64_t* chars_capacity,
                          or_status* st) {
  memset(st, 0, sizeof *st);
  st->first_error_offset = UINT64_MAX;
  csv_out o = {n_cols, col_types, defaults, out_offsets, out_chars, out_typed, records_capacity,
               chars_capacity, st, NULL, 0, 0};
  for (int c = 0; c < n_cols; c++)
    if (col_types[c] == C_STR && out_offsets[c]) out_offsets[c][0] = 0;
  /* the current record: its value bytes in one buffer, a list of fields */
  uint8_t* rbytes = NULL;
  size_t rb_len = 0, rb_cap = 0;
  or_field* fields = NULL;
  size_t nf = 0, nf_cap = 0;
  uint64_t rec_in = 0;   /* records read (index in the input) */
  uint64_t rec_out = 0;  /* records emitted */
  uint64_t skip_i = 0;   /* next entry of skip_records */
  int s = EOR, tag = T_RD;
  uint64_t field_start = 0;
#define PUSH_FIELD()                                                          \
  do {                                                                        \
    if (nf == nf_cap) {                                                       \
      nf_cap = nf_cap ? 2 * nf_cap : 16;                                      \
      fields = (or_field*)realloc(fields, nf_cap * sizeof *fields);           \
    }                                                                         \
    fields[nf].start = field_start;                                           \
    fields[nf].vbeg = vbeg;                                                   \
    fields[nf].vlen = rb_len - vbeg;                                          \
    nf++;                                                                     \
  } while (0)
  uint64_t vbeg = 0;
  /* emit (or drop) the collected record whose terminator is at off */
#define CLOSE_RECORD(off)                                                     \
  do {                                                                        \
    while (skip_i < n_skip_records && skip_records[skip_i] < rec_in) skip_i++; \
    const int skipped = skip_i < n_skip_records && skip_records[skip_i] == rec_in; \
    const int bad = (int)nf != n_cols;                                        \
    if (skipped) {                                                            \
      st->n_dropped++;                                                        \
    } else if (bad && reject) {                                               \
      flag(st, E_COLCOUNT, (off), 1);                                         \
      st->n_dropped++;                                                        \
    } else {                                                                  \
      for (size_t f = 0; f < nf; f++) {                                       \
        o.val_len = 0;                                                        \
        for (uint64_t k = 0; k < fields[f].vlen; k++)                         \
          field_value_push(&o, rbytes[fields[f].vbeg + k]);                   \
        close_field(&o, rec_out, (int)f, fields[f].start);                    \
      }                                                                       \
      close_record(&o, rec_out, (int)nf - 1, (off));                          \
      rec_out++;                                                              \
    }                                                                         \
    rec_in++;                                                                 \
    nf = 0; rb_len = 0; vbeg = 0;                                             \
  } while (0)
  /* one symbol [i, j) at a time; a symbol's offsets (terminator, invalid
   * transition) are those of its last byte */
  for (uint64_t i = 0, j; i < n; i = j) {
    uint32_t sym;
    j = sym_at(in, n, enc, i, &sym);
    s = csv_step(&y, s, sym, &tag);
    switch (tag) {
      case T_DATA:
        for (uint64_t k = i; k < j; k++) {
          if (rb_len == rb_cap) {
            rb_cap = rb_cap ? 2 * rb_cap : 256;
            rbytes = (uint8_t*)realloc(rbytes, rb_cap);
          }
          rbytes[rb_len++] = in[k];
        }
        break;
      case T_CTRL: break;
      case T_FD:
        PUSH_FIELD();
        vbeg = rb_len; field_start = j;
        break;
      case T_RD:
        PUSH_FIELD();
        CLOSE_RECORD(j - 1);
        field_start = j;
        break;
      default:
        flag(st, E_INVALID_INPUT, j - 1, 1);
        break;
    }
  }
  if (s == INV || !csv_accepting(s)) {
    /* the input ends inside a record that never closes (the automaton
     * died, or ended in a non-accepting state): the fields the record
     * closed are converted as they closed (unless the record is skipped);
     * nothing else of it forms a field */
    if (s != INV) flag(st, E_BAD_END_STATE, n, 1);
    while (skip_i < n_skip_records && skip_records[skip_i] < rec_in) skip_i++;
    if (!(skip_i < n_skip_records && skip_records[skip_i] == rec_in))
      for (size_t f = 0; f < nf; f++) {
        o.val_len = 0;
        for (uint64_t k = 0; k < fields[f].vlen; k++) field_value_push(&o, rbytes[fields[f].vbeg + k]);
        close_field(&o, rec_out, (int)f, fields[f].start);
      }
  } else if (n > 0 && tag != T_RD) {            /* unterminated last record */
    PUSH_FIELD();
    CLOSE_RECORD(n);
  }
#undef PUSH_FIELD
#undef CLOSE_RECORD
  st->n_records = rec_out;
  free(o.val);
  free(rbytes);
  free(fields);
  return 0;
}

int or_csv_parse_ex(const uint8_t* in, uint64_t n, uint8_t fd, uint8_t rd, uint8_t q, int crlf,
                    int n_cols, const int32_t* col_types, const uint64_t* defaults, int reject,
                    const uint64_t* skip_records, uint64_t n_skip_records,
                    int32_t** out_offsets, uint8_t** out_chars, void** out_typed,
                    uint64_t records_capacity, const uint64_t* chars_capacity, or_status* st) {
  return csv_parse_core(in, n, 0, syms_of(crlf ? 2 : 0, fd, rd, q), n_cols, col_types, defaults,
                        reject, skip_records, n_skip_records, out_offsets, out_chars, out_typed,
                        records_capacity, chars_capacity, st);
}

/* The quoted-CSV parse of an input in a variable-length encoding (enc 1
 * UTF-8, 2 UTF-16LE; ParPaRaw Section 3.4): the DFA reads symbols, with
 * field delimiter, record delimiter and quote given as code points. */
int or_csv_parse_enc(const uint8_t* in, uint64_t n, int enc, uint32_t fd, uint32_t rd, uint32_t q,
                     int n_cols, const int32_t* col_types, const uint64_t* defaults, int reject,
                     const uint64_t* skip_records, uint64_t n_skip_records,
                     int32_t** out_offsets, uint8_t** out_chars, void** out_typed,
                     uint64_t records_capacity, const uint64_t* chars_capacity, or_status* st) {
  const csv_syms y = {fd, rd, q, -1};
  return csv_parse_core(in, n, enc, y, n_cols, col_types, defaults, reject, skip_records,
                        n_skip_records, out_offsets, out_chars, out_typed, records_capacity,
                        chars_capacity, st);
}

int or_csv_parse(const uint8_t* in, uint64_t n, uint8_t fd, uint8_t rd, uint8_t q, int crlf,
                 int n_cols, const int32_t* col_types, int32_t** out_offsets,
                 uint8_t** out_chars, void** out_typed, uint64_t records_capacity,
                 const uint64_t* chars_capacity, or_status* st) {
  return or_csv_parse_ex(in, n, fd, rd, q, crlf, n_cols, col_types, NULL, 0, NULL, 0,
                         out_offsets, out_chars, out_typed, records_capacity, chars_capacity, st);
}

/* Numeric type inference (ParPaRaw Section 4, "Type inference"): the
 * smallest type that backs a field's value, in the order int8 < int32 <
 * int64 < float64 < string (codes 1..5; 0: an empty field, which constrains
 * nothing).  An integer beyond int64 is backed by float64. */
static int field_type(const uint8_t* v, size_t n) {
  if (n == 0) return 0;
  int64_t x;
  int rc = conv_int(v, n, -128, 127, &x);
  if (rc == 0) return 1;
  if (rc == E_NUM_OVERFLOW) {
    if (conv_int(v, n, INT32_MIN, INT32_MAX, &x) == 0) return 2;
    if (conv_int(v, n, INT64_MIN, INT64_MAX, &x) == 0) return 3;
    return 4;
  }
  double d;
  if (conv_f64(v, n, &d) == 0) return 4;
  return 5;
}

/* Per column c < n_cols, the largest field_type over the input's records
 * (fields past n_cols are ignored, a missing field is empty); a column
 * whose fields are all empty gets int8.  out[c] holds the library's column
 * codes: 1 int8, 2 int32, 3 int64, 4 float64, 0 string. */
void or_infer_types(const uint8_t* in, uint64_t n, uint8_t fd, uint8_t rd, uint8_t q, int crlf,
                    int n_cols, int32_t* out, or_status* st) {
  memset(st, 0, sizeof *st);
  st->first_error_offset = UINT64_MAX;
  int best[64];
  for (int c = 0; c < n_cols; c++) best[c] = 0;
  csv_syms y = syms_of(crlf ? 2 : 0, fd, rd, q);
  uint8_t* val = NULL;
  size_t len = 0, cap = 0;
  int s = EOR, tag = T_RD, col = 0;
  uint64_t rec = 0;
  for (uint64_t i = 0; i <= n; i++) {
    const int end = i == n;
    if (!end) {
      s = csv_step(&y, s, in[i], &tag);
      if (tag == T_DATA) {
        if (len == cap) { cap = cap ? 2 * cap : 256; val = (uint8_t*)realloc(val, cap); }
        val[len++] = in[i];
        continue;
      }
      if (tag == T_CTRL) continue;
      if (tag != T_FD && tag != T_RD) { flag(st, E_INVALID_INPUT, i, 1); continue; }
    } else if (s == INV || !csv_accepting(s) || n == 0 || tag == T_RD) {
      if (s != INV && !csv_accepting(s)) flag(st, E_BAD_END_STATE, n, 1);
      break;
    }
    if (col < n_cols) {
      const int t = field_type(val, len);
      if (t > best[col]) best[col] = t;
    }
    len = 0;
    if (end || tag == T_RD) { rec++; col = 0; } else col++;
  }
  static const int32_t code[6] = {1, 1, 2, 3, 4, 0};
  for (int c = 0; c < n_cols; c++) out[c] = code[best[c]];
  st->n_records = rec;
  free(val);
}

/* Rows are lines: the bytes up to and including each record-delimiter byte
 * (rd), whatever the quoting (ParPaRaw Section 4, "Skipping rows": a record
 * may span several rows), plus a last line without one.  Copies the input
 * without the rows listed in skip_rows (sorted ascending) to out; returns
 * the bytes written. */
uint64_t or_skip_rows(const uint8_t* in, uint64_t n, uint8_t rd, const uint64_t* skip_rows,
                      uint64_t n_skip_rows, uint8_t* out) {
  uint64_t row = 0, w = 0, k = 0;
  for (uint64_t i = 0; i < n; i++) {
    while (k < n_skip_rows && skip_rows[k] < row) k++;
    if (!(k < n_skip_rows && skip_rows[k] == row)) out[w++] = in[i];
    if (in[i] == rd) row++;
  }
  return w;
}

/* ------------------------------------------------------------ tokenize */
int or_tokenize(const uint8_t* in, uint64_t n, uint8_t* out_id, uint64_t* out_start,
                uint32_t* out_len, uint64_t cap, or_status* st) {
  memset(st, 0, sizeof *st);
  st->first_error_offset = UINT64_MAX;
  int s = L_START;
  uint64_t k = 0, cur_start = 0;
  for (uint64_t i = 0; i < n; i++) {
    int begin, before = s;
    s = lex_step(s, in[i], &begin);
    if (s == L_INV && before != L_INV) flag(st, E_INVALID_INPUT, i, 1);
    if (i == 0 || begin) {
      if (i > 0) {               /* close the previous token */
        if (k - 1 < cap) {
          out_id[k - 1] = (uint8_t)lex_token_id(before, in[cur_start]);
          out_len[k - 1] = (uint32_t)(i - cur_start);
        }
      }
      if (k < cap) out_start[k] = i;
      else flag(st, E_CAPACITY, 0, 0);
      k++;
      cur_start = i;
    }
  }
  if (n > 0 && k - 1 < cap) {
    out_id[k - 1] = (uint8_t)lex_token_id(s, in[cur_start]);
    out_len[k - 1] = (uint32_t)(n - cur_start);
  }
  if (s != L_INV && !lex_accepting(s)) flag(st, E_BAD_END_STATE, n, 1);
  st->n_tokens = k;
  return 0;
}

/* ------------------------------------------- the method's own steps */
/* These restate ParPaRaw Section 3.1 (multi-instance DFA, state-transition
 * vectors, composite operation, exclusive scan) and Section 3.2 (absolute /
 * relative column offsets) directly, for the tests to compare with the
 * sequential walk above.                                                  */

/* State-transition vector of one chunk: entry i = the final state of the
 * DFA instance that started the chunk in state i (Figure 2).              */
/* Column-count inference (ParPaRaw Section 4, "Inferring or validating
 * number of columns"; inputs may hold records with varying numbers of field
 * delimiters): the fewest and the most fields of any record, walking the
 * DFA byte by byte.  A record has one more field than
 * field delimiters; a non-empty tail without a record delimiter is one more
 * record.  out[0] = min, out[1] = max (both 0 without records); st gets
 * n_records and the same data errors as the parse (invalid input, a
 * non-accepting end state).                                              */
void or_count_fields(const uint8_t* in, uint64_t n, uint8_t fd, uint8_t rd, uint8_t q, int crlf,
                     uint64_t* out, or_status* st) {
  memset(st, 0, sizeof *st);
  st->first_error_offset = UINT64_MAX;
  csv_syms y = syms_of(crlf ? 2 : 0, fd, rd, q);
  int s = EOR, tag = T_RD;
  uint64_t fields = 1, mn = UINT64_MAX, mx = 0, recs = 0;
  for (uint64_t i = 0; i < n; i++) {
    s = csv_step(&y, s, in[i], &tag);
    if (tag == T_INVALID) { flag(st, E_INVALID_INPUT, i, 1); break; }
    if (tag == T_FD) fields++;
    if (tag == T_RD) {
      if (fields < mn) mn = fields;
      if (fields > mx) mx = fields;
      recs++;
      fields = 1;
    }
  }
  if (!(st->error & E_INVALID_INPUT)) {
    if (!csv_accepting(s)) flag(st, E_BAD_END_STATE, n, 1);
    if (n > 0 && tag != T_RD) {  /* the open tail is one more record */
      if (fields < mn) mn = fields;
      if (fields > mx) mx = fields;
      recs++;
    }
  }
  out[0] = recs ? mn : 0;
  out[1] = recs ? mx : 0;
  st->n_records = recs;
}

void or_stv(int kind, uint8_t fd, uint8_t rd, uint8_t q, const uint8_t* chunk,
            uint64_t len, uint8_t* stv) {
  csv_syms y = syms_of(kind, fd, rd, q);
  for (int i = 0; i < nstates(kind); i++) {
    int s = i, t;
    for (uint64_t j = 0; j < len; j++) s = step_any(kind, &y, s, chunk[j], &t);
    stv[i] = (uint8_t)s;
  }
}

/* Composite operation: (a o b)[i] = b[a[i]] with a the earlier chunk —
 * running a's chunk from state i and then b's chunk from where it ended.   */
void or_compose(int ns, const uint8_t* a, const uint8_t* b, uint8_t* out) {
  for (int i = 0; i < ns; i++) out[i] = b[a[i]];
}

/* Chunk start states by the scan: STVs per chunk, exclusive composite scan
 * seeded with the identity vector, start state = prefix[start state].      */
void or_chunk_start_states(int kind, uint8_t fd, uint8_t rd, uint8_t q,
                           const uint8_t* in, uint64_t n, uint64_t chunk, uint8_t* out) {
  int ns = nstates(kind), s0 = 0;
  uint8_t pre[16], stv[16], tmp[16];
  for (int i = 0; i < ns; i++) pre[i] = (uint8_t)i;   /* identity */
  uint64_t c = 0;
  for (uint64_t off = 0; off < n; off += chunk, c++) {
    out[c] = pre[s0];
    uint64_t len = n - off < chunk ? n - off : chunk;
    or_stv(kind, fd, rd, q, in + off, len, stv);
    or_compose(ns, pre, stv, tmp);
    memcpy(pre, tmp, (size_t)ns);
  }
}

/* Column offset of one chunk (Section 3.2, Figure 4): absolute when the
 * chunk holds a record delimiter (then the number of field delimiters after
 * the last record delimiter), else relative (the number of field
 * delimiters).  Tags come from running the DFA from the chunk's start. */
void or_colofs_chunk(const uint8_t* tags, uint64_t len, int* is_abs, uint64_t* o) {
  *is_abs = 0; *o = 0;
  for (uint64_t j = 0; j < len; j++) {
    if (tags[j] == T_RD) { *is_abs = 1; *o = 0; }
    else if (tags[j] == T_FD) (*o)++;
  }
}
/* Column-offset operator: b absolute wins; b relative adds to a. */
void or_colofs_combine(int a_abs, uint64_t a_o, int b_abs, uint64_t b_o, int* abs_out,
                       uint64_t* o_out) {
  if (b_abs) { *abs_out = 1; *o_out = b_o; }
  else { *abs_out = a_abs; *o_out = a_o + b_o; }
}

/* Column-count inference per chunk (ParPaRaw Section 4, "Inferring or
 * validating number of columns"): whether the chunk has a record delimiter,
 * the field delimiters before its first one (the relative count, all of
 * them without one), the fewest and most fields of the records that start
 * after its first record delimiter and end at a later one, and the field
 * delimiters after its last one.                                          */
typedef struct { int has_rd; uint64_t pre, post, mn, mx; } or_fagg;
static void or_fields_chunk(const uint8_t* tags, uint64_t len, or_fagg* a) {
  uint64_t run = 0;
  a->has_rd = 0; a->pre = a->post = 0; a->mn = UINT64_MAX; a->mx = 0;
  for (uint64_t j = 0; j < len; j++) {
    if (tags[j] == T_FD) { run++; continue; }
    if (tags[j] != T_RD) continue;
    if (!a->has_rd) a->pre = run;
    else {
      if (run + 1 < a->mn) a->mn = run + 1;
      if (run + 1 > a->mx) a->mx = run + 1;
    }
    a->has_rd = 1;
    run = 0;
  }
  if (a->has_rd) a->post = run; else a->pre = run;
}
/* Chunk a followed by chunk b: the record across the seam, when both sides
 * close it, has a.post + b.pre + 1 fields.                               */
static void or_fields_combine(const or_fagg* a, const or_fagg* b, or_fagg* o) {
  or_fagg r;
  if (!a->has_rd && !b->has_rd) {
    r = *a; r.pre = a->pre + b->pre;
  } else if (!a->has_rd) {
    r = *b; r.pre = a->pre + b->pre;
  } else if (!b->has_rd) {
    r = *a; r.post = a->post + b->pre;
  } else {
    uint64_t mid = a->post + b->pre + 1;
    r.has_rd = 1; r.pre = a->pre; r.post = b->post;
    r.mn = a->mn < b->mn ? a->mn : b->mn; if (mid < r.mn) r.mn = mid;
    r.mx = a->mx > b->mx ? a->mx : b->mx; if (mid > r.mx) r.mx = mid;
  }
  *o = r;
}

/* Brute force over every string of length 1..max_len on `alpha`: for every
 * chunk size 1..max_len, the scan-derived chunk start states must equal the
 * sequential walk's state at each chunk start, the scanned column offsets
 * must equal the sequential column index, and (CSV, strings without an
 * invalid byte) the chunks' column-count aggregates combined in order must
 * give the sequential walk's fewest and most fields per record.  Returns
 * the number of mismatches; *checked = strings visited.                   */
uint64_t or_bruteforce(int kind, uint8_t fd, uint8_t rd, uint8_t q, const uint8_t* alpha,
                       int n_alpha, int max_len, uint64_t* checked) {
  uint64_t bad = 0;
  *checked = 0;
  uint8_t str[16], seq_state[17], tags[16], starts[16];
  int idx[16];
  csv_syms y = syms_of(kind, fd, rd, q);
  for (int len = 1; len <= max_len; len++) {
    for (int i = 0; i < len; i++) idx[i] = 0;
    for (;;) {
      for (int i = 0; i < len; i++) str[i] = alpha[idx[i]];
      /* sequential walk */
      int s = 0, t;
      uint64_t col_seq[17];
      uint64_t col = 0;
      for (int i = 0; i < len; i++) {
        seq_state[i] = (uint8_t)s;
        col_seq[i] = col;
        s = step_any(kind, &y, s, str[i], &t);
        tags[i] = (uint8_t)t;
        if (is_csv(kind)) { if (t == T_RD) col = 0; else if (t == T_FD) col++; }
      }
      (*checked)++;
      /* sequential fewest / most fields per record (valid strings) */
      int valid = 1;
      uint64_t f = 1, smn = UINT64_MAX, smx = 0;
      for (int i = 0; i < len; i++) {
        if (tags[i] == T_INVALID) valid = 0;
        if (tags[i] == T_FD) f++;
        if (tags[i] == T_RD) { if (f < smn) smn = f; if (f > smx) smx = f; f = 1; }
      }
      if (tags[len - 1] != T_RD) { if (f < smn) smn = f; if (f > smx) smx = f; }
      for (int ch = 1; ch <= max_len; ch++) {
        or_chunk_start_states(kind, fd, rd, q, str, (uint64_t)len, (uint64_t)ch, starts);
        int nch = (len + ch - 1) / ch;
        int a_abs = 1; uint64_t a_o = 0;         /* seed: absolute column 0 */
        or_fagg fa = {1, 0, 0, UINT64_MAX, 0};   /* seed: a record ends before the input */
        for (int c = 0; c < nch; c++) {
          if (starts[c] != seq_state[c * ch]) bad++;
          if (is_csv(kind)) {
            if (!a_abs || a_o != col_seq[c * ch]) bad++;
            int b_abs; uint64_t b_o;
            int clen = len - c * ch < ch ? len - c * ch : ch;
            or_colofs_chunk(tags + c * ch, (uint64_t)clen, &b_abs, &b_o);
            or_colofs_combine(a_abs, a_o, b_abs, b_o, &a_abs, &a_o);
            or_fagg fb;
            or_fields_chunk(tags + c * ch, (uint64_t)clen, &fb);
            or_fields_combine(&fa, &fb, &fa);
          }
        }
        if (is_csv(kind) && valid) {
          uint64_t mn = fa.mn, mx = fa.mx;
          if (tags[len - 1] != T_RD) {         /* the open tail is one more record */
            if (fa.post + 1 < mn) mn = fa.post + 1;
            if (fa.post + 1 > mx) mx = fa.post + 1;
          }
          if (mn != smn || mx != smx) bad++;
        }
      }
      int p = len - 1;
      while (p >= 0 && ++idx[p] == n_alpha) { idx[p] = 0; p--; }
      if (p < 0) break;
    }
  }
  return bad;
}
