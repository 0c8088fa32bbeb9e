/*
 * Seeded synthetic inputs for the five workloads of the delimiter-separated
 * parser and the JSON-like lexer.  This module only *writes* text; it holds
 * none of the parsing method's arithmetic, so both the CPU oracle and the GPU
 * path may consume what it produces.
 *
 * Random numbers: splitmix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), written from its published
 * definition: add the golden-gamma increment, then two xor-shift-multiply
 * mixing rounds and a final xor-shift.
 *
 * Every generator appends whole records (or whole top-level values for the
 * token stream) while the total stays <= the byte target, so the CSV inputs
 * always end with the record delimiter.
 *
 * Optional record start offsets (byte offset of every record / top-level
 * value), and per-column totals of the value bytes written.
 *
 * Optional sidecar (ground truth, for small inputs):
 *   CSV:    every field's value text, unescaped, followed by one 0x00 byte,
 *           fields in record-major order.
 *   tokens: per token 1 byte kind + 4 bytes little-endian length.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  uint64_t n_bytes;      /* bytes written                                   */
  uint64_t n_records;    /* CSV records                                     */
  uint64_t n_fields;     /* CSV fields                                      */
  uint64_t n_tokens;     /* lexer tokens (whitespace runs included)         */
  uint64_t quoted_bytes; /* bytes from an opening quote to its closing one  */
  uint64_t side_len;     /* sidecar bytes written                           */
  int32_t side_overflow; /* 1 if the sidecar buffer was too small           */
  int32_t pad;
  uint64_t col_value_bytes[64]; /* per column: bytes of the values written
                                   (unescaped), summed over all records     */
} dg_info;

/* ---------------------------------------------------------------- rng */
typedef struct { uint64_t s; } rng_t;

static inline uint64_t sm64(rng_t* r) {
  uint64_t z = (r->s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
/* uniform integer in [0, m) by the multiply-high reduction */
static inline uint64_t below(rng_t* r, uint64_t m) {
  return (uint64_t)(((unsigned __int128)sm64(r) * m) >> 64);
}
static inline int64_t uni(rng_t* r, int64_t lo, int64_t hi) { /* inclusive */
  return lo + (int64_t)below(r, (uint64_t)(hi - lo + 1));
}
static inline double u01(rng_t* r) { return (double)(sm64(r) >> 11) * 0x1.0p-53; }
static inline int chance(rng_t* r, double p) { return u01(r) < p; }
static double normal(rng_t* r) { /* Box-Muller */
  double u1 = u01(r), u2 = u01(r);
  if (u1 < 1e-300) u1 = 1e-300;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* ---------------------------------------------------------------- sinks */
typedef struct {
  uint8_t* buf; uint64_t len, cap;   /* record scratch                   */
  uint64_t colbytes[64];             /* value bytes per column, this record */
  uint8_t* side; uint64_t slen, scap; int soverflow;
  uint64_t quoted;                   /* quoted bytes in this record      */
  uint64_t fields;
} rec_t;

static inline void put(rec_t* w, uint8_t c) {
  if (w->len < w->cap) w->buf[w->len] = c;
  w->len++;
}
static inline void puts_n(rec_t* w, const char* s, size_t n) {
  for (size_t i = 0; i < n; i++) put(w, (uint8_t)s[i]);
}
static inline void sput(rec_t* w, uint8_t c) {
  if (!w->side) return;
  if (w->slen < w->scap) w->side[w->slen++] = c; else w->soverflow = 1;
}
static inline void sput_n(rec_t* w, const char* s, size_t n) {
  for (size_t i = 0; i < n; i++) sput(w, (uint8_t)s[i]);
}

static const char ALNUM[] =
    "ABCDEFGHIJKLMNOPQRSTUVWXYZabcdefghijklmnopqrstuvwxyz0123456789";
static const char ALNUM_SP[] =
    "ABCDEFGHIJKLMNOPQRSTUVWXYZabcdefghijklmnopqrstuvwxyz0123456789 ";
static const char ALNUM_SP_DOT[] =
    "ABCDEFGHIJKLMNOPQRSTUVWXYZabcdefghijklmnopqrstuvwxyz0123456789 .";

static int fmt_u64(char* o, uint64_t v) {
  char t[24]; int n = 0;
  do { t[n++] = (char)('0' + v % 10); v /= 10; } while (v);
  for (int i = 0; i < n; i++) o[i] = t[n - 1 - i];
  return n;
}
static int fmt_i64(char* o, int64_t v) {
  if (v < 0) { o[0] = '-'; return 1 + fmt_u64(o + 1, (uint64_t)(-(v + 1)) + 1); }
  return fmt_u64(o, (uint64_t)v);
}

/* A field whose text is written verbatim (no quoting). */
static void field_plain(rec_t* w, const char* s, size_t n) {
  puts_n(w, s, n); sput_n(w, s, n); sput(w, 0);
  if (w->fields < 64) w->colbytes[w->fields] += n;
  w->fields++;
}

/* A quoted field: body chars given unescaped; '"' is doubled in the output. */
static void field_quoted(rec_t* w, const char* body, size_t n) {
  put(w, '"'); w->quoted += 1;
  for (size_t i = 0; i < n; i++) {
    if (body[i] == '"') { put(w, '"'); put(w, '"'); w->quoted += 2; }
    else { put(w, (uint8_t)body[i]); w->quoted += 1; }
  }
  put(w, '"'); w->quoted += 1;
  sput_n(w, body, n); sput(w, 0);
  if (w->fields < 64) w->colbytes[w->fields] += n;
  w->fields++;
}

/* Body of a quoted field with embedded specials: per char 70 % from the
 * alphabet, 10 % each of ',', '\n', '"'; at least one special when n > 0. */
static void special_body(rng_t* r, char* b, size_t n, const char* alpha, size_t na) {
  int any = 0;
  for (size_t i = 0; i < n; i++) {
    uint64_t k = below(r, 10);
    if (k < 7) b[i] = alpha[below(r, na)];
    else { b[i] = (k == 7) ? ',' : (k == 8) ? '\n' : '"'; any = 1; }
  }
  if (n && !any) {
    static const char sp[3] = {',', '\n', '"'};
    b[below(r, n)] = sp[below(r, 3)];
  }
}

/* ------------------------------------------------------------ workloads */
/* Workload 1: 4 string columns, length U{1..12} over [A-Za-z0-9];
 * 10 % of fields quoted with embedded delimiters and doubled quotes. */
static void rec_w1(rng_t* r, rec_t* w, uint64_t idx) {
  (void)idx;
  char b[16];
  for (int c = 0; c < 4; c++) {
    size_t n = (size_t)uni(r, 1, 12);
    if (chance(r, 0.10)) { special_body(r, b, n, ALNUM, 62); field_quoted(w, b, n); }
    else { for (size_t i = 0; i < n; i++) b[i] = ALNUM[below(r, 62)]; field_plain(w, b, n); }
    put(w, c == 3 ? '\n' : ',');
  }
}

/* Workload 2: 16 columns, types i f s i f s i f s i f s i i s s. */
static const char W2_TYPES[16] = {'i','f','s','i','f','s','i','f','s','i','f','s','i','i','s','s'};
static void rec_w2(rng_t* r, rec_t* w, uint64_t idx) {
  (void)idx;
  char b[64];
  for (int c = 0; c < 16; c++) {
    char t = W2_TYPES[c];
    if (t == 'i') {
      int n = fmt_i64(b, uni(r, -1000000000LL, 1000000000LL));
      field_plain(w, b, (size_t)n);
    } else if (t == 'f') {
      int n = snprintf(b, sizeof b, "%.6g", normal(r) * 1e3);
      field_plain(w, b, (size_t)n);
    } else {
      size_t n = (size_t)uni(r, 0, 32);
      if (chance(r, 0.05)) { special_body(r, b, n, ALNUM_SP, 63); field_quoted(w, b, n); }
      else { for (size_t i = 0; i < n; i++) b[i] = ALNUM_SP[below(r, 63)]; field_plain(w, b, n); }
    }
    put(w, c == 15 ? '\n' : ',');
  }
}

/* Workload 3: int32 id, long text (lognormal length, mean 600, max 8192),
 * int8 score in 1..5.  Quoted texts carry ~1 % each of ',', '\n', '"'. */
static char* W3_BODY;
static void rec_w3(rng_t* r, rec_t* w, uint64_t idx) {
  char b[24];
  int n = fmt_u64(b, idx);
  field_plain(w, b, (size_t)n);
  put(w, ',');
  double len = exp((log(600.0) - 0.5) + normal(r));
  size_t L = len < 1.0 ? 1 : len > 8192.0 ? 8192 : (size_t)len;
  if (chance(r, 0.87)) {
    for (size_t i = 0; i < L; i++) {
      uint64_t k = below(r, 100);
      W3_BODY[i] = k == 0 ? ',' : k == 1 ? '\n' : k == 2 ? '"' : ALNUM_SP_DOT[below(r, 64)];
    }
    field_quoted(w, W3_BODY, L);
  } else {
    for (size_t i = 0; i < L; i++) W3_BODY[i] = ALNUM_SP_DOT[below(r, 64)];
    field_plain(w, W3_BODY, L);
  }
  put(w, ',');
  b[0] = (char)('0' + uni(r, 1, 5));
  field_plain(w, b, 1);
  put(w, '\n');
}

/* Workload 4: 18 unquoted columns ts ts i f i f i f i f i f i f i i i i;
 * timestamps uniform over 2020..2025, ints 0..9, floats %.2f of U[0,500]. */
static void civil(int64_t days, int* y, int* m, int* d) {
  /* days since 1970-01-01 -> proleptic Gregorian date (era arithmetic) */
  days += 719468;
  int64_t era = (days >= 0 ? days : days - 146096) / 146097;
  int64_t doe = days - era * 146097;
  int64_t yoe = (doe - doe / 1460 + doe / 36524 - doe / 146096) / 365;
  int64_t yy = yoe + era * 400;
  int64_t doy = doe - (365 * yoe + yoe / 4 - yoe / 100);
  int64_t mp = (5 * doy + 2) / 153;
  *d = (int)(doy - (153 * mp + 2) / 5 + 1);
  *m = (int)(mp < 10 ? mp + 3 : mp - 9);
  *y = (int)(yy + (*m <= 2));
}
static void two(char* o, int v) { o[0] = (char)('0' + v / 10); o[1] = (char)('0' + v % 10); }
static void rec_w4(rng_t* r, rec_t* w, uint64_t idx) {
  (void)idx;
  static const int64_t T0 = 1577836800LL;   /* 2020-01-01 00:00:00 UTC */
  static const int64_t T1 = 1767225599LL;   /* 2025-12-31 23:59:59 UTC */
  char b[32];
  for (int c = 0; c < 18; c++) {
    if (c < 2) {
      int64_t t = uni(r, T0, T1);
      int y, mo, d;
      civil(t / 86400, &y, &mo, &d);
      int64_t s = t % 86400;
      b[0] = (char)('0' + y / 1000); b[1] = (char)('0' + (y / 100) % 10);
      two(b + 2, y % 100); b[4] = '-'; two(b + 5, mo); b[7] = '-'; two(b + 8, d);
      b[10] = ' '; two(b + 11, (int)(s / 3600)); b[13] = ':'; two(b + 14, (int)(s / 60 % 60));
      b[16] = ':'; two(b + 17, (int)(s % 60));
      field_plain(w, b, 19);
    } else if (c >= 14 || (c % 2) == 0) {
      b[0] = (char)('0' + uni(r, 0, 9));
      field_plain(w, b, 1);
    } else {
      int64_t cents = uni(r, 0, 50000);
      int n = fmt_u64(b, (uint64_t)(cents / 100));
      b[n] = '.'; two(b + n + 1, (int)(cents % 100));
      field_plain(w, b, (size_t)n + 3);
    }
    put(w, c == 17 ? '\n' : ',');
  }
}

/* ------------------------------------------------------ JSON-like stream */
enum { K_LBRACE = 0, K_RBRACE, K_LBRACK, K_RBRACK, K_COMMA, K_COLON,
       K_STRING, K_INT, K_FLOAT, K_WS };

typedef struct { rec_t* w; rng_t* r; uint64_t tokens; int budget; } jctx;

static void tok(jctx* j, int kind, uint64_t start) {
  rec_t* w = j->w;
  uint32_t len = (uint32_t)(w->len - start);
  sput(w, (uint8_t)kind);
  sput(w, (uint8_t)len); sput(w, (uint8_t)(len >> 8));
  sput(w, (uint8_t)(len >> 16)); sput(w, (uint8_t)(len >> 24));
  j->tokens++;
}
static void jws(jctx* j) { /* optional whitespace run between tokens */
  if (!chance(j->r, 0.3)) return;
  static const char WS[4] = {' ', '\t', '\n', '\r'};
  uint64_t s = j->w->len;
  int n = (int)uni(j->r, 1, 8);
  for (int i = 0; i < n; i++) put(j->w, (uint8_t)WS[below(j->r, 4)]);
  tok(j, K_WS, s);
}
static void jpunct(jctx* j, char c, int kind) {
  uint64_t s = j->w->len; put(j->w, (uint8_t)c); tok(j, kind, s);
}
static void jstring(jctx* j, int maxlen) {
  static const char HEX[] = "0123456789abcdefABCDEF";
  static const char PR[] =
      "ABCDEFGHIJKLMNOPQRSTUVWXYZabcdefghijklmnopqrstuvwxyz0123456789 _-.:/#@";
  rec_t* w = j->w; rng_t* r = j->r;
  uint64_t s = w->len;
  put(w, '"');
  int n = (int)uni(r, 0, maxlen);
  for (int i = 0; i < n; i++) {
    if (chance(r, 0.1)) {
      put(w, '\\');
      switch (below(r, 5)) {
        case 0: put(w, '"'); break;
        case 1: put(w, '\\'); break;
        case 2: put(w, 'n'); break;
        case 3: put(w, 't'); break;
        default:
          put(w, 'u');
          for (int k = 0; k < 4; k++) put(w, (uint8_t)HEX[below(r, 22)]);
      }
    } else {
      put(w, (uint8_t)PR[below(r, sizeof(PR) - 1)]);
    }
  }
  put(w, '"');
  tok(j, K_STRING, s);
}
static void jint(jctx* j) {
  char b[24];
  uint64_t s = j->w->len;
  int n = fmt_i64(b, uni(j->r, -1000000000LL, 1000000000LL));
  puts_n(j->w, b, (size_t)n);
  tok(j, K_INT, s);
}
static void jfloat(jctx* j) {
  rec_t* w = j->w; rng_t* r = j->r;
  uint64_t s = w->len;
  int digits = (int)uni(r, 1, 17);
  if (chance(r, 0.5)) put(w, '-');
  if (chance(r, 0.5)) {           /* fixed notation: int part '.' frac  */
    int ip = (int)uni(r, 1, digits > 6 ? 6 : digits);
    int fp = digits - ip; if (fp < 1) fp = 1;
    if (ip == 1) put(w, (uint8_t)('0' + below(r, 10)));
    else { put(w, (uint8_t)('1' + below(r, 9)));
           for (int i = 1; i < ip; i++) put(w, (uint8_t)('0' + below(r, 10))); }
    put(w, '.');
    for (int i = 0; i < fp; i++) put(w, (uint8_t)('0' + below(r, 10)));
  } else {                        /* exponent notation, %.*e style      */
    put(w, (uint8_t)('1' + below(r, 9)));
    if (digits > 1) {
      put(w, '.');
      for (int i = 1; i < digits; i++) put(w, (uint8_t)('0' + below(r, 10)));
    }
    put(w, chance(r, 0.8) ? 'e' : 'E');
    uint64_t k = below(r, 3);
    if (k == 0) put(w, '+'); else if (k == 1) put(w, '-');
    int ex = (int)uni(r, 0, 308);
    char b[8]; int n = fmt_u64(b, (uint64_t)ex);
    if (n == 1 && chance(r, 0.5)) put(w, '0');
    puts_n(w, b, (size_t)n);
  }
  tok(j, K_FLOAT, s);
}
static void jvalue(jctx* j, int depth);
static void jobject(jctx* j, int depth) {
  jpunct(j, '{', K_LBRACE);
  int n = (int)uni(j->r, 0, 5);
  for (int i = 0; i < n; i++) {
    if (i) { jws(j); jpunct(j, ',', K_COMMA); }
    jws(j); jstring(j, 12); jws(j); jpunct(j, ':', K_COLON); jws(j);
    jvalue(j, depth + 1);
  }
  jws(j);
  jpunct(j, '}', K_RBRACE);
}
static void jarray(jctx* j, int depth) {
  jpunct(j, '[', K_LBRACK);
  int n = (int)uni(j->r, 0, 5);
  for (int i = 0; i < n; i++) {
    if (i) { jws(j); jpunct(j, ',', K_COMMA); }
    jws(j);
    jvalue(j, depth + 1);
  }
  jws(j);
  jpunct(j, ']', K_RBRACK);
}
static void jvalue(jctx* j, int depth) {
  j->budget--;
  double u = u01(j->r);
  if (depth < 6 && j->budget > 0 && u < 0.22) { jobject(j, depth); return; }
  if (depth < 6 && j->budget > 0 && u < 0.32) { jarray(j, depth); return; }
  uint64_t k = below(j->r, 3);
  if (k == 0) jstring(j, 40); else if (k == 1) jint(j); else jfloat(j);
}
/* Workload 5: one top-level object per "record", whitespace between them. */
static uint64_t W5_TOKENS;
static void rec_w5(rng_t* r, rec_t* w, uint64_t idx) {
  (void)idx;
  jctx j = {w, r, 0, 400};
  jobject(&j, 1);
  uint64_t s = w->len;
  int n = (int)uni(r, 1, 8);
  static const char WS[4] = {' ', '\t', '\n', '\r'};
  for (int i = 0; i < n; i++) put(w, (uint8_t)WS[below(r, 4)]);
  tok(&j, K_WS, s);
  W5_TOKENS = j.tokens;
}

/* ------------------------------------------------------------- driver */
typedef void (*rec_fn)(rng_t*, rec_t*, uint64_t);

int dg_generate(int cfg, uint64_t target, uint64_t seed, uint8_t* out, uint64_t cap,
                uint8_t* side, uint64_t side_cap, dg_info* info, uint64_t* rec_offsets,
                uint64_t rec_offsets_cap) {
  rec_fn fn;
  switch (cfg) {
    case 1: fn = rec_w1; break;
    case 2: fn = rec_w2; break;
    case 3: fn = rec_w3; break;
    case 4: fn = rec_w4; break;
    case 5: fn = rec_w5; break;
    default: return -1;
  }
  if (target > cap) target = cap;
  memset(info, 0, sizeof *info);
  const uint64_t RCAP = 1u << 24;           /* one record / top-level value */
  uint8_t* rb = (uint8_t*)malloc(RCAP);
  W3_BODY = (char*)malloc(8192 + 16);
  if (!rb || !W3_BODY) { free(rb); free(W3_BODY); return -2; }
  rng_t r = {seed};
  uint64_t pos = 0, idx = 0;
  rec_t w;
  memset(&w, 0, sizeof w);
  w.buf = rb; w.cap = RCAP; w.side = side; w.scap = side_cap;
  for (;;) {
    uint64_t slen0 = w.slen;
    w.len = 0; w.quoted = 0; w.fields = 0; W5_TOKENS = 0;
    memset(w.colbytes, 0, sizeof w.colbytes);
    fn(&r, &w, idx);
    if (w.len > RCAP) { free(rb); free(W3_BODY); return -3; }
    if (pos + w.len > target) { w.slen = slen0; break; }
    memcpy(out + pos, rb, w.len);
    if (rec_offsets && idx < rec_offsets_cap) rec_offsets[idx] = pos;
    for (int c = 0; c < 64; c++) info->col_value_bytes[c] += w.colbytes[c];
    pos += w.len;
    info->quoted_bytes += w.quoted;
    info->n_fields += w.fields;
    info->n_tokens += W5_TOKENS;
    idx++;
  }
  info->n_bytes = pos;
  info->n_records = cfg == 5 ? 0 : idx;
  info->side_len = w.slen;
  info->side_overflow = w.soverflow;
  free(rb); free(W3_BODY);
  return 0;
}
