// libpp C ABI: argument checks, DFA descriptor builders and launch glue.
// Every entry point validates its arguments on the host, allocates the
// cross-block scan scratch stream-ordered (cudaMallocAsync / cudaFreeAsync
// on the caller's stream) and enqueues its kernels; nothing synchronises.
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_internal.h"

namespace ppi {

cudaError_t current_device(int* dev) {
  const cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  return (*dev >= 0 && *dev < MAX_DEVICES) ? cudaSuccess : cudaErrorInvalidDevice;
}

cudaError_t sm_count(int* out) {
  static DeviceOnce once;
  static int n_sm[MAX_DEVICES];
  int dev;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return e;
  e = once.run(dev, [](int d) {
    return cudaDeviceGetAttribute(&n_sm[d], cudaDevAttrMultiProcessorCount, d);
  });
  if (e == cudaSuccess) *out = n_sm[dev];
  return e;
}

uint32_t g_spin_limit = 1u << 22;  // ~1 s of polling before a look-back gives up
uint32_t g_withhold = 0;           // test hook, see pp_debug_set_withhold

// Stage timing for benchmarks: events of the recorded calls, up to
// PP_STAGES + 1 per call, and how many of them each call recorded.
constexpr int STAGE_EVENTS = PP_STAGES + 1;
cudaEvent_t* g_stage_ev = nullptr;
int* g_stage_n = nullptr;
int g_stage_cap = 0, g_stage_used = 0, g_stage_cur = -1;

bool stage_begin() {
  g_stage_cur = g_stage_used < g_stage_cap ? g_stage_used++ : -1;
  return g_stage_cur >= 0;
}
void stage_mark(int k, cudaStream_t stream) {
  if (g_stage_cur < 0 || k >= STAGE_EVENTS) return;
  cudaEventRecord(g_stage_ev[g_stage_cur * STAGE_EVENTS + k], stream);
  if (k + 1 > g_stage_n[g_stage_cur]) g_stage_n[g_stage_cur] = k + 1;
}
}

namespace {

using ppi::GenericDfa;

pp_rc cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return PP_OK;
  if (e == cudaErrorMemoryAllocation) return PP_ENOMEM;
  return PP_ECUDA;
}

// Structural checks shared by all DFA consumers.
bool dfa_ok(const pp_dfa_desc* d, int max_states) {
  if (!d) return false;
  if (d->n_states < 1 || d->n_states > max_states || d->n_groups < 1 || d->n_groups > PP_MAX_GROUPS)
    return false;
  if (d->start_state >= d->n_states) return false;
  if (d->invalid_state != 0xFF && d->invalid_state >= d->n_states) return false;
  if (d->start_state == d->invalid_state) return false;
  for (int b = 0; b < 256; ++b)
    if (d->byte_to_group[b] >= d->n_groups) return false;
  if (d->encoding > PP_ENC_UTF16LE || d->n_syms > PP_MAX_SYMS) return false;
  for (int k = 0; k < d->n_syms; ++k) {
    const uint32_t cp = d->sym_cp[k];
    if (cp < 0x80 || cp > 0x10FFFF || (cp >= 0xD800 && cp <= 0xDFFF)) return false;
    if (d->sym_group[k] >= d->n_groups) return false;
    for (int j = 0; j < k; ++j)
      if (d->sym_cp[j] == cp) return false;
  }
  for (int g = 0; g < d->n_groups; ++g)
    for (int s = 0; s < d->n_states; ++s) {
      if (d->delta[g][s] >= d->n_states) return false;
      if (d->tag[s][g] > PP_TAG_BEGIN) return false;
    }
  if (d->invalid_state != 0xFF)
    for (int g = 0; g < d->n_groups; ++g)
      if (d->delta[g][d->invalid_state] != d->invalid_state) return false;  // absorbing
  return true;
}

GenericDfa to_generic(const pp_dfa_desc* d) {
  GenericDfa g;
  std::memset(&g, 0, sizeof g);
  g.n_states = d->n_states;
  g.start_state = d->start_state;
  g.invalid_state = d->invalid_state;
  g.accept_mask = d->accept_mask;
  std::memcpy(g.byte_to_group, d->byte_to_group, 256);
  std::memcpy(g.delta, d->delta, sizeof g.delta);
  std::memcpy(g.tag, d->tag, sizeof g.tag);
  std::memcpy(g.token_id, d->token_id, sizeof g.token_id);
  std::memcpy(g.byte_token_id, d->byte_token_id, sizeof g.byte_token_id);
  return g;
}

// LUT entry of one symbol group for pp_parse (see parse_kernel):
//   bits  0..15  nibble s = delta[g][s], s = 0..3 (byte-permute selector)
//   bits 16..19  4: the invalid state maps to itself
//   bits 20..27  2-bit tag of (s, g), s = 0..3: DATA 0, FD 1, RD 2, CTRL 3
//   bits 28..29  3: the invalid state's bytes are treated as control
//   bit  30      the group is not inert in the sticky state X: it changes
//                X or tags a byte of X other than DATA
//   bit  31      the group is not the background group
uint32_t parse_lut_entry(const pp_dfa_desc* d, int g, int x) {
  uint32_t e = 4u << 16 | 3u << 28;
  for (int s = 0; s < 4; ++s) {
    const uint32_t nx = s < d->n_states ? d->delta[g][s] : uint32_t(s);
    e |= nx << (4 * s);
    uint32_t tg = 0;
    if (s < d->n_states) {
      switch (d->tag[s][g]) {
        case PP_TAG_FD: tg = 1; break;
        case PP_TAG_RD: tg = 2; break;
        case PP_TAG_CTRL: tg = 3; break;
        default: tg = 0; break;
      }
    }
    e |= tg << (20 + 2 * s);
  }
  if (g != d->background_group) e |= 1u << 31;
  if (x < 4 && (d->delta[g][x] != x || d->tag[x][g] != PP_TAG_DATA)) e |= 1u << 30;
  return e;
}

// LUT entry of a byte of a multi-byte symbol of group g other than its
// last: it keeps the state and is tagged CTRL where the symbol is a
// delimiter or control symbol, else DATA; never background.
uint32_t parse_lut_mid_entry(const pp_dfa_desc* d, int g, int x) {
  uint32_t e = 4u << 16 | 3u << 28 | 1u << 31;
  for (int s = 0; s < 4; ++s) {
    e |= uint32_t(s) << (4 * s);
    const int t = s < d->n_states ? d->tag[s][g] : PP_TAG_DATA;
    if (t == PP_TAG_FD || t == PP_TAG_RD || t == PP_TAG_CTRL) e |= 3u << (20 + 2 * s);
  }
  if (x < 4) {
    const int t = d->tag[x][g];
    if (t == PP_TAG_FD || t == PP_TAG_RD || t == PP_TAG_CTRL) e |= 1u << 30;
  }
  return e;
}

// The live state with the fewest non-inert symbol groups (a group is inert
// in s if it keeps s and tags the byte DATA); runs of inert bytes in that
// state need no DFA steps.  4 when no state has an inert group.
int sticky_state(const pp_dfa_desc* d) {
  const int live = d->n_states == 5 ? 4 : d->n_states;
  int best = 4, best_n = d->n_groups;
  for (int s = 0; s < live; ++s) {
    int n = 0;
    for (int g = 0; g < d->n_groups; ++g)
      if (d->delta[g][s] != s || d->tag[s][g] != PP_TAG_DATA) ++n;
    if (n < best_n) { best = s; best_n = n; }
  }
  return best;
}

// pp_parse's extra constraints: at most 4 live states plus an absorbing
// invalid state with index 4; INVALID tags exactly on transitions into it;
// no BEGIN tags; a valid background group (idempotent transition, value
// bytes only) when one is named.
bool parse_dfa_ok(const pp_dfa_desc* d) {
  if (!dfa_ok(d, 5)) return false;
  if (d->n_states == 5 && d->invalid_state != 4) return false;
  if (d->n_states < 5 && d->invalid_state != 0xFF) return false;
  const int live = d->n_states == 5 ? 4 : d->n_states;
  for (int g = 0; g < d->n_groups; ++g)
    for (int s = 0; s < live; ++s) {
      const bool to_inv = d->delta[g][s] == d->invalid_state;
      const int tg = d->tag[s][g];
      if (tg == PP_TAG_BEGIN) return false;
      if ((tg == PP_TAG_INVALID) != to_inv) return false;
    }
  const int bg = d->background_group;
  if (bg != 0xFF) {
    if (bg >= d->n_groups) return false;
    for (int s = 0; s < d->n_states; ++s) {
      const int s1 = d->delta[bg][s];
      if (d->delta[bg][s1] != s1) return false;  // idempotent
      if (s == d->invalid_state) continue;
      const int tg = d->tag[s][bg];
      if (tg != PP_TAG_DATA && tg != PP_TAG_INVALID) return false;
    }
  }
  return true;
}

}  // namespace

namespace ppi {

bool generic_dfa_ok(const pp_dfa_desc* d) {
  return dfa_ok(d, PP_MAX_STATES) && d->encoding == PP_ENC_BYTES;
}
GenericDfa to_generic_dfa(const pp_dfa_desc* d) { return to_generic(d); }

// Host half of pp_parse: checks the arguments and fills the kernel
// parameters (everything but the scratch carve).
pp_rc parse_prepare(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                    const pp_coltype* col_types, int32_t* const out_offsets[],
                    uint8_t* const out_chars[], void* const out_typed[],
                    size_t records_capacity, const size_t chars_capacity[],
                    pp_status* d_status, ParseParams* out) {
  ParseParams& p = *out;
  if (!d_status || (n_bytes && !d_in) || !parse_dfa_ok(dfa)) return PP_EINVAL;
  if (n_cols < 1 || n_cols > PP_MAX_COLS || !col_types) return PP_EINVAL;
  std::memset(&p, 0, sizeof p);
  int n_str = 0;
  bool any_out = false;
  for (int c = 0; c < n_cols; ++c) {
    const int ty = col_types[c];
    if (ty < PP_COL_STRING || ty > PP_COL_TIMESTAMP) return PP_EINVAL;
    if (ty == PP_COL_TIMESTAMP && dfa->encoding != PP_ENC_BYTES) return PP_EINVAL;
    p.coltype[c] = uint8_t(ty);
    p.stridx[c] = -1;
    if (ty == PP_COL_STRING) {
      if (n_str >= ppi::MAX_STR_COLS) return PP_EINVAL;
      p.stridx[c] = int8_t(n_str);
      p.strcol[n_str] = uint8_t(c);
      p.strmask |= 1ull << c;
      ++n_str;
    }
    if ((out_offsets && out_offsets[c]) || (out_chars && out_chars[c]) ||
        (out_typed && out_typed[c]))
      any_out = true;
  }
  for (int c = n_cols; c < PP_MAX_COLS; ++c) { p.coltype[c] = PP_COL_SKIP; p.stridx[c] = -1; }
  if (any_out) {
    for (int c = 0; c < n_cols; ++c) {
      const int ty = col_types[c], si = p.stridx[c];
      if (ty == PP_COL_STRING) {
        if (!out_offsets || !out_chars || !out_offsets[c] || !chars_capacity) return PP_EINVAL;
        if (!out_chars[c] && chars_capacity[c]) return PP_EINVAL;
        p.offsets[si] = out_offsets[c];
        p.chars[si] = out_chars[c];
        p.chars_cap[si] = chars_capacity[c];
      } else if (ty != PP_COL_SKIP) {
        if (!out_typed || (!out_typed[c] && records_capacity)) return PP_EINVAL;
        p.typed[c] = out_typed[c];
      }
    }
    p.rec_cap = records_capacity;
  } else {
    p.rec_cap = ~0ull;
    for (int c = 0; c < n_str; ++c) p.chars_cap[c] = ~0ull;
  }
  p.in = d_in;
  p.n = n_bytes;
  // positions and record counts travel in 40 bits through the tile pass's look-back
  if (uint64_t(n_bytes) >= (1ull << 40)) return PP_ETOOLARGE;
  const uint64_t tile = ppi::parse_tile_bytes();
  const uint64_t nt = (uint64_t(n_bytes) + tile - 1) / tile;
  if (nt > 0xFFFFFFF0ull) return PP_EINVAL;
  p.n_tiles = uint32_t(nt);
  p.spin_limit = ppi::g_spin_limit;
  p.dbg_withhold = ppi::g_withhold;
  const int x = sticky_state(dfa);
  p.sticky = uint32_t(x);
  if (dfa->encoding == PP_ENC_BYTES) {
    for (int b = 0; b < 256; ++b) p.lut[b] = parse_lut_entry(dfa, dfa->byte_to_group[b], x);
  } else {
    // LUT rows by symbol code: a one-byte symbol below 0x80 is its own code,
    // SYM_LAST + g the last byte of a longer symbol of group g, SYM_MID + g
    // its other bytes
    const int dflt = dfa->byte_to_group[0x80];
    for (int b = 0; b < 256; ++b) p.lut[b] = parse_lut_entry(dfa, dflt, x);
    for (int b = 0; b < 0x80; ++b) p.lut[b] = parse_lut_entry(dfa, dfa->byte_to_group[b], x);
    for (int g = 0; g < dfa->n_groups; ++g) {
      p.lut[SYM_LAST + g] = parse_lut_entry(dfa, g, x);
      p.lut[SYM_MID + g] = parse_lut_mid_entry(dfa, g, x);
    }
    p.enc = dfa->encoding;
    p.sym_n = dfa->n_syms;
    p.sym_dflt = uint8_t(dflt);
    for (int b = 0; b < 0x80; ++b) p.sym_b2g[b] = dfa->byte_to_group[b];
    for (int k = 0; k < dfa->n_syms; ++k) {
      p.sym_cp[k] = dfa->sym_cp[k];
      p.sym_g[k] = dfa->sym_group[k];
    }
  }
  p.bg_next = 0;
  if (dfa->background_group != 0xFF) {
    for (int s = 0; s < 4; ++s)
      p.bg_next |= uint32_t(s < dfa->n_states ? dfa->delta[dfa->background_group][s] : s)
                   << (4 * s);
    p.bg_next |= 4u << 16;
  }
  p.accept_mask = dfa->accept_mask;
  p.start_state = dfa->start_state;
  p.has_inv = dfa->invalid_state == 4;
  p.n_cols = n_cols;
  p.n_str = n_str;
  p.has_out = any_out ? 1 : 0;
  p.st = d_status;
  return PP_OK;
}

}  // namespace ppi

extern "C" {

const char* pp_strerror(int code) {
  switch (code) {
    case PP_OK: return "ok";
    case PP_EINVAL: return "invalid argument";
    case PP_ECUDA: return "CUDA error";
    case PP_ENOMEM: return "out of device memory";
    case PP_ETOOLARGE: return "input needs more scratch than the fixed buffer holds";
    case PP_ECHUNK: return "a record is longer than the streaming chunk";
    default: return "unknown error";
  }
}

size_t pp_tile_bytes(void) { return ppi::parse_tile_bytes(); }

pp_rc pp_desc_csv(pp_dfa_desc* out, uint8_t fd, uint8_t rd, uint8_t quote) {
  if (!out || fd == rd || fd == quote || rd == quote) return PP_EINVAL;
  std::memset(out, 0, sizeof *out);
  enum { EOR = 0, FLD = 1, ENC = 2, ESC = 3, INV = 4 };
  enum { GQ = 0, GF = 1, GR = 2, GO = 3 };
  out->n_states = 5;
  out->n_groups = 4;
  out->start_state = EOR;
  out->invalid_state = INV;
  out->accept_mask = (1u << EOR) | (1u << FLD) | (1u << ESC);
  out->background_group = GO;
  for (int b = 0; b < 256; ++b) out->byte_to_group[b] = GO;
  out->byte_to_group[quote] = GQ;
  out->byte_to_group[fd] = GF;
  out->byte_to_group[rd] = GR;
  // one row per symbol group: next state for EOR, FLD, ENC, ESC, INV
  static const uint8_t next[4][5] = {
      /* quote */ {ENC, INV, ESC, ENC, INV},
      /* fd    */ {EOR, EOR, ENC, EOR, INV},
      /* rd    */ {EOR, EOR, ENC, EOR, INV},
      /* other */ {FLD, FLD, ENC, INV, INV},
  };
  static const uint8_t tags[4][5] = {
      /* quote */ {PP_TAG_CTRL, PP_TAG_INVALID, PP_TAG_CTRL, PP_TAG_DATA, PP_TAG_INVALID},
      /* fd    */ {PP_TAG_FD, PP_TAG_FD, PP_TAG_DATA, PP_TAG_FD, PP_TAG_INVALID},
      /* rd    */ {PP_TAG_RD, PP_TAG_RD, PP_TAG_DATA, PP_TAG_RD, PP_TAG_INVALID},
      /* other */ {PP_TAG_DATA, PP_TAG_DATA, PP_TAG_DATA, PP_TAG_INVALID, PP_TAG_INVALID},
  };
  for (int g = 0; g < 4; ++g)
    for (int s = 0; s < 5; ++s) {
      out->delta[g][s] = next[g][s];
      out->tag[s][g] = tags[g][s];
    }
  for (int s = 0; s < PP_MAX_STATES; ++s) out->token_id[s] = 255;
  for (int b = 0; b < 256; ++b) out->byte_token_id[b] = 255;
  return PP_OK;
}

pp_rc pp_desc_csv_enc(pp_dfa_desc* out, int encoding, uint32_t fd, uint32_t rd, uint32_t quote) {
  if (!out || (encoding != PP_ENC_UTF8 && encoding != PP_ENC_UTF16LE)) return PP_EINVAL;
  const uint32_t cps[3] = {quote, fd, rd};  // groups 0, 1, 2 as in pp_desc_csv
  for (int k = 0; k < 3; ++k)
    if (cps[k] > 0x10FFFF || (cps[k] >= 0xD800 && cps[k] <= 0xDFFF)) return PP_EINVAL;
  if (fd == rd || fd == quote || rd == quote) return PP_EINVAL;
  // the byte descriptor with placeholder symbols, then the real ones
  pp_rc rc = pp_desc_csv(out, 0, 1, 2);
  if (rc != PP_OK) return rc;
  for (int b = 0; b < 3; ++b) out->byte_to_group[b] = 3;  // the catch-all group
  out->encoding = uint8_t(encoding);
  for (int k = 0; k < 3; ++k) {
    if (cps[k] < 0x80) {
      out->byte_to_group[cps[k]] = uint8_t(k);
    } else {
      out->sym_cp[out->n_syms] = cps[k];
      out->sym_group[out->n_syms] = uint8_t(k);
      ++out->n_syms;
    }
  }
  return PP_OK;
}

pp_rc pp_desc_csv_crlf(pp_dfa_desc* out, uint8_t fd, uint8_t quote) {
  const uint8_t lf = 0x0A, cr = 0x0D;
  if (!out || fd == lf || fd == cr || quote == lf || quote == cr) return PP_EINVAL;
  const pp_rc rc = pp_desc_csv(out, fd, lf, quote);
  if (rc != PP_OK) return rc;
  // a fifth symbol group for CR: a control symbol outside quotes that
  // leaves the field open, data inside quotes
  enum { EOR = 0, FLD = 1, ENC = 2, ESC = 3, INV = 4 };
  const int GC = 4;
  out->n_groups = 5;
  out->byte_to_group[cr] = GC;
  static const uint8_t next[5] = {FLD, FLD, ENC, FLD, INV};
  static const uint8_t tags[5] = {PP_TAG_CTRL, PP_TAG_CTRL, PP_TAG_DATA, PP_TAG_CTRL,
                                  PP_TAG_INVALID};
  for (int s = 0; s < 5; ++s) {
    out->delta[GC][s] = next[s];
    out->tag[s][GC] = tags[s];
  }
  return PP_OK;
}

pp_rc pp_desc_json_lexer(pp_dfa_desc* out) {
  if (!out) return PP_EINVAL;
  std::memset(out, 0, sizeof *out);
  enum { START, WS, PUNCT, STR_OPEN, STR, STR_BSL, STR_END, NEG, ZERO, INT, DOT, FRAC, EXP_E,
         EXP_SIGN, EXP, INV };
  enum { G_WS, G_PUNCT, G_QUOTE, G_BSL, G_MINUS, G_PLUS, G_ZERO, G_D19, G_DOT, G_E, G_OTHER };
  out->n_states = 16;
  out->n_groups = 11;
  out->start_state = START;
  out->invalid_state = INV;
  out->background_group = 0xFF;
  out->accept_mask = (1u << START) | (1u << WS) | (1u << PUNCT) | (1u << STR_END) | (1u << ZERO) |
                     (1u << INT) | (1u << FRAC) | (1u << EXP);
  for (int b = 0; b < 256; ++b) out->byte_to_group[b] = G_OTHER;
  for (const char* p = " \t\n\r"; *p; ++p) out->byte_to_group[uint8_t(*p)] = G_WS;
  for (const char* p = "{}[],:"; *p; ++p) out->byte_to_group[uint8_t(*p)] = G_PUNCT;
  out->byte_to_group[uint8_t('"')] = G_QUOTE;
  out->byte_to_group[uint8_t('\\')] = G_BSL;
  out->byte_to_group[uint8_t('-')] = G_MINUS;
  out->byte_to_group[uint8_t('+')] = G_PLUS;
  out->byte_to_group[uint8_t('0')] = G_ZERO;
  for (int c = '1'; c <= '9'; ++c) out->byte_to_group[c] = G_D19;
  out->byte_to_group[uint8_t('.')] = G_DOT;
  out->byte_to_group[uint8_t('e')] = G_E;
  out->byte_to_group[uint8_t('E')] = G_E;

  // the state that begins a token on each group (INV: none)
  static const uint8_t begin_of[11] = {WS, PUNCT, STR_OPEN, INV, NEG, INV, ZERO, INT, INV, INV, INV};
  for (int s = 0; s < 16; ++s)
    for (int g = 0; g < 11; ++g) {
      const bool digit = g == G_ZERO || g == G_D19;
      const bool ends_number = g == G_WS || g == G_PUNCT || g == G_QUOTE || g == G_MINUS;
      uint8_t nx = INV;
      bool begins = false;
      switch (s) {
        case START: case WS: case PUNCT: case STR_END:
          nx = begin_of[g];
          begins = nx != INV && !(s == WS && g == G_WS);
          break;
        case STR_OPEN: case STR:
          nx = g == G_QUOTE ? STR_END : g == G_BSL ? STR_BSL : STR;
          break;
        case STR_BSL: nx = STR; break;
        case NEG: nx = g == G_ZERO ? ZERO : g == G_D19 ? INT : INV; break;
        case ZERO: case INT: case FRAC: case EXP:
          if (ends_number) { nx = begin_of[g]; begins = true; }
          else if (s == ZERO) nx = g == G_DOT ? DOT : g == G_E ? EXP_E : INV;
          else if (s == INT) nx = digit ? INT : g == G_DOT ? DOT : g == G_E ? EXP_E : INV;
          else if (s == FRAC) nx = digit ? FRAC : g == G_E ? EXP_E : INV;
          else nx = digit ? EXP : INV;
          break;
        case DOT: nx = digit ? FRAC : INV; break;
        case EXP_E: nx = (g == G_PLUS || g == G_MINUS) ? EXP_SIGN : digit ? EXP : INV; break;
        case EXP_SIGN: nx = digit ? EXP : INV; break;
        default: nx = INV; break;
      }
      out->delta[g][s] = nx;
      out->tag[s][g] = nx == INV ? PP_TAG_INVALID : begins ? PP_TAG_BEGIN : PP_TAG_DATA;
    }
  for (int s = 0; s < PP_MAX_STATES; ++s) out->token_id[s] = 255;
  out->token_id[WS] = 9;
  out->token_id[PUNCT] = 0xFE;
  out->token_id[STR_END] = 6;
  out->token_id[ZERO] = 7;
  out->token_id[INT] = 7;
  out->token_id[FRAC] = 8;
  out->token_id[EXP] = 8;
  for (int b = 0; b < 256; ++b) out->byte_token_id[b] = 255;
  const char* punct = "{}[],:";
  for (int i = 0; punct[i]; ++i) out->byte_token_id[uint8_t(punct[i])] = uint8_t(i);
  return PP_OK;
}

pp_rc pp_parse(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
               const pp_coltype* col_types, int32_t* const out_offsets[],
               uint8_t* const out_chars[], void* const out_typed[], size_t records_capacity,
               const size_t chars_capacity[], pp_status* d_status, cudaStream_t stream) {
  ppi::ParseParams p;
  const pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, n_cols, col_types, out_offsets,
                                      out_chars, out_typed, records_capacity, chars_capacity,
                                      d_status, &p);
  if (rc != PP_OK) return rc;
  const int ns = ppi::parse_ns_width(p.n_str);
  const size_t sb = ppi::parse_scratch_bytes(p.n_tiles, ns, p.enc != 0);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, sb, stream);
  if (e != cudaSuccess) return cuda_rc(e);
  ppi::parse_scratch_carve(scratch, p.n_tiles, ns, &p.s, p.enc != 0);
  e = ppi::launch_parse(p, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

pp_rc pp_debug_parse_tags(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                          uint32_t* d_bits, pp_status* d_status, cudaStream_t stream) {
  if (!d_bits && n_bytes) return PP_EINVAL;
  const pp_coltype skip = PP_COL_SKIP;
  ppi::ParseParams p;
  const pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, 1, &skip, nullptr, nullptr, nullptr, 0,
                                      nullptr, d_status, &p);
  if (rc != PP_OK) return rc;
  p.dbg_tags = d_bits;
  const int ns = ppi::parse_ns_width(p.n_str);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, ppi::parse_scratch_bytes(p.n_tiles, ns, p.enc != 0),
                                  stream);
  if (e != cudaSuccess) return cuda_rc(e);
  ppi::parse_scratch_carve(scratch, p.n_tiles, ns, &p.s, p.enc != 0);
  e = ppi::launch_parse(p, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

pp_rc pp_count_fields(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                      uint64_t* d_fields, pp_status* d_status, cudaStream_t stream) {
  if (!d_fields || (dfa && dfa->encoding != PP_ENC_BYTES)) return PP_EINVAL;
  if (n_bytes > (size_t(1) << 36)) return PP_ETOOLARGE;  // the tile reduction's 32-bit ranges
  const pp_coltype skip = PP_COL_SKIP;
  ppi::ParseParams p;
  const pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, 1, &skip, nullptr, nullptr, nullptr, 0,
                                      nullptr, d_status, &p);
  if (rc != PP_OK) return rc;
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, ppi::fields_scratch_bytes(p.n_tiles), stream);
  if (e != cudaSuccess) return cuda_rc(e);
  e = ppi::launch_count_fields(p, scratch, d_fields, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

pp_rc pp_tokenize(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                  uint8_t* out_token_id, uint64_t* out_start, uint32_t* out_len,
                  size_t tokens_capacity, pp_status* d_status, cudaStream_t stream) {
  if (!d_status || (n_bytes && !d_in) || !ppi::generic_dfa_ok(dfa)) return PP_EINVAL;
  if (tokens_capacity && (!out_token_id || !out_start || !out_len)) return PP_EINVAL;
  const GenericDfa g = to_generic(dfa);
  const size_t sb = ppi::tokenize_scratch_bytes(n_bytes);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, sb, stream);
  if (e != cudaSuccess) return cuda_rc(e);
  e = ppi::launch_tokenize(d_in, n_bytes, g, out_token_id, out_start, out_len, tokens_capacity,
                           d_status, scratch, sb, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

pp_rc pp_tags(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, uint8_t* d_state_before,
              uint8_t* d_tag, pp_status* d_status, cudaStream_t stream) {
  if (!d_status || (n_bytes && (!d_in || !d_state_before || !d_tag)) ||
      !ppi::generic_dfa_ok(dfa))
    return PP_EINVAL;
  const GenericDfa g = to_generic(dfa);
  const size_t sb = ppi::tags_scratch_bytes(n_bytes);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, sb, stream);
  if (e != cudaSuccess) return cuda_rc(e);
  e = ppi::launch_tags(d_in, n_bytes, g, d_state_before, d_tag, d_status, scratch, sb, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (e == cudaSuccess) e = ef;
  return cuda_rc(e);
}

pp_rc pp_count_byte(const uint8_t* d_in, size_t n_bytes, uint8_t value, uint64_t* d_count,
                    cudaStream_t stream) {
  if (!d_count || (n_bytes && !d_in)) return PP_EINVAL;
  return cuda_rc(ppi::launch_count_byte(d_in, n_bytes, value, d_count, stream));
}

void pp_debug_set_spin_limit(uint32_t polls) { ppi::g_spin_limit = polls ? polls : (1u << 22); }

void pp_debug_set_withhold(int on) { ppi::g_withhold = on ? 1u : 0u; }

pp_rc pp_debug_stage_timing(int n_calls) {
  using namespace ppi;
  for (int i = 0; i < g_stage_cap * STAGE_EVENTS; ++i) cudaEventDestroy(g_stage_ev[i]);
  delete[] g_stage_ev;
  delete[] g_stage_n;
  g_stage_ev = nullptr;
  g_stage_n = nullptr;
  g_stage_cap = g_stage_used = 0;
  g_stage_cur = -1;
  if (n_calls <= 0) return PP_OK;
  g_stage_n = new int[n_calls]();
  g_stage_ev = new cudaEvent_t[size_t(n_calls) * STAGE_EVENTS];
  for (int i = 0; i < n_calls * STAGE_EVENTS; ++i) {
    if (cudaEventCreate(&g_stage_ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_stage_ev[j]);
      delete[] g_stage_ev;
      delete[] g_stage_n;
      g_stage_ev = nullptr;
      g_stage_n = nullptr;
      return PP_ECUDA;
    }
  }
  g_stage_cap = n_calls;
  return PP_OK;
}

int pp_debug_stage_ms(float* out, int max_calls) {
  using namespace ppi;
  const int n = g_stage_used < max_calls ? g_stage_used : max_calls;
  for (int i = 0; i < n; ++i) {
    cudaEvent_t* e = g_stage_ev + i * STAGE_EVENTS;
    const int marks = g_stage_n[i];
    for (int k = 0; k < PP_STAGES; ++k) out[PP_STAGES * i + k] = 0.f;
    if (marks < 2) continue;
    if (cudaEventSynchronize(e[marks - 1]) != cudaSuccess) return -1;
    for (int k = 0; k + 1 < marks; ++k)
      if (cudaEventElapsedTime(&out[PP_STAGES * i + k], e[k], e[k + 1]) != cudaSuccess) return -1;
  }
  return n;
}

}  // extern "C"
