// pp_parse: DFA-based parsing of delimiter-separated input into Arrow-style
// columns on sm_103a.
//
// The input is cut into 16 KiB tiles; each worker thread of the tile pass
// owns a 32-byte chunk (one bit per byte in the bitmap indexes).
//
// 0. Tile start states (tile_stv_kernel, tile_state_kernel).  A warp per
//    tile folds the tile's transition vector (ParPaRaw Section 3.1, Figure
//    2): the vector of the four live states sits in one register, one byte
//    per state, and each byte composes it with its symbol group's row by
//    one byte-permute (the row-per-group transition table of ParPaRaw
//    Section 5, Table 1, read from a per-lane replicated shared-memory LUT).
//    An exclusive composite scan over tiles gives every tile's true start
//    state.
// 1. Tile pass (parse_kernel).  Tiles reach shared memory by a 1-D bulk copy
//    (TMA engine), the next tile's copy running while the current one is
//    processed.  Per tile: chunk vectors composed across the block give every
//    chunk's start state; one DFA per thread tags its chunk (the three bitmap
//    indexes of Section 3.1); record counts and absolute/relative column
//    offsets (Section 3.2, Figure 4) are scanned over the tile and then across
//    tiles by a decoupled look-back run by a dedicated context warp, and the
//    value bytes per string column by a chars warp; each lane walks its
//    chunk's fields into a column-major (column, record) slot table in shared
//    memory; string value bytes are compacted per column into shared memory
//    (stream compaction in place of ParPaRaw's radix partitioning, Section
//    3.3) and written as 16-byte stores, and one lane per field writes the
//    Arrow offset or converts the number (Section 3.3), 32 consecutive rows
//    of a column to a warp for coalesced stores.  Each input byte is read
//    twice from HBM (once per pass) and every output byte written once; no
//    per-byte intermediate reaches HBM.  The kernel is instantiated plain
//    (byte inputs, every record emitted) and general (encodings, the options
//    of pp_parse_ex, type inference, streamed chunks).
// 2. Long numeric fields (long_field_kernel): fields over 256 bytes, queued
//    by the tile pass, converted by a warp each (Section 3.3's collaboration
//    on long fields).
// Column-count inference (fields_kernel, fields_reduce_kernel) reuses the
// tile start states.
#include <cstdint>
#include <cuda_runtime.h>
#include <algorithm>

#include "pp.h"
#include "pp_device.cuh"
#include "pp_internal.h"
#include "pp_numeric.cuh"
#include "pp_stv16.cuh"

namespace {
using namespace ppd;
using ppi::ParseParams;

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int CB = 32;                 // bytes per thread chunk (one bitmap word)
constexpr int TILE = NT * CB;          // 16 KiB
constexpr int STAGE_BYTES = TILE + 16 * (ppi::MAX_STR_COLS + 1);
constexpr int LUT_BYTES = 256 * 32 * 4;
constexpr int SLOT_CAP = 4096;         // (column, record) slots per pass
constexpr uint32_t ABS32 = 1u << 31;
constexpr uint32_t SLOT_DEFAULT = 0xFFFFFFFDu; // missing field: column default
constexpr uint32_t WAIT_LIMIT = 1u << 24;      // bounded mbarrier polls

// ------------------------------------------------------------ helpers
// (record count, column offset, last terminator) of a byte range; column
// offset: bit 31 = absolute, else relative; last: ((pos+1) << 8) | state
// after the terminator, 0 = none.
struct V2 { uint32_t rec, col, last; };

__device__ __forceinline__ V2 op2_32(V2 a, V2 b) {
  V2 o;
  o.rec = a.rec + b.rec;
  o.col = (b.col & ABS32) ? b.col : ((a.col & ABS32) | ((a.col + b.col) & ~ABS32));
  o.last = b.last ? b.last : a.last;
  return o;
}
__device__ __forceinline__ V2 shfl_up_v2(V2 v, int d) {
  return {__shfl_up_sync(FULL, v.rec, d), __shfl_up_sync(FULL, v.col, d),
          __shfl_up_sync(FULL, v.last, d)};
}
template <int K>
struct AddOp {
  __device__ void operator()(const uint64_t (&a)[K], const uint64_t (&b)[K],
                             uint64_t (&o)[K]) const {
#pragma unroll
    for (int k = 0; k < K; ++k) o[k] = a[k] + b[k];
  }
};

// packed 16-bit counters: string column si lives in word si/4, lane si%4
template <int NSW>
__device__ __forceinline__ void add16(uint64_t (&c)[NSW], int si, uint32_t v) {
#pragma unroll
  for (int k = 0; k < NSW; ++k)
    if (k == (si >> 2)) c[k] += uint64_t(v) << (16 * (si & 3));
}
template <int NSW>
__device__ __forceinline__ uint32_t get16(const uint64_t (&c)[NSW], int si) {
  uint64_t w = 0;
#pragma unroll
  for (int k = 0; k < NSW; ++k)
    if (k == (si >> 2)) w = c[k];
  return uint32_t(w >> (16 * (si & 3))) & 0xFFFFu;
}

// byte p of the tile (linear layout in shared memory)
__device__ __forceinline__ uint32_t tile_byte(const uint8_t* tile_s, uint32_t p) { return tile_s[p]; }
__device__ __forceinline__ uint32_t popc_range(const uint32_t* m, uint32_t a, uint32_t b) {
  uint32_t n = 0;
  while (a < b) {
    const uint32_t w = a >> 5, lo = a & 31u;
    const uint32_t hi = min(b - (w << 5), 32u);
    n += __popc(m[w] & range_mask(lo, hi));
    a = (w + 1) << 5;
  }
  return n;
}

// ------------------------------------------------ symbols of an encoding
// Inputs in UTF-8 or UTF-16LE (ParPaRaw Section 3.4): a symbol may span
// several bytes and cross chunk and tile boundaries.  Every byte gets a code
// that indexes the LUT in place of the byte: the symbol's transition is
// taken at its last byte (code: the byte for a one-byte symbol below 0x80,
// else SYM_LAST + its group); its other bytes keep the state and take the
// symbol's tag as DATA or CTRL (code SYM_MID + group).  So the bytes at a
// chunk's start that continue a symbol begun before it change nothing, as
// the page asks, and a multi-byte delimiter's other bytes drop out of the
// values like control bytes.  Symbol boundaries: in UTF-8 a byte that is
// not 0b10xxxxxx with the 0b10xxxxxx bytes after it; in UTF-16LE 2-byte
// units from the input's first byte, a high surrogate and the low
// surrogate after it forming one symbol.  B(q) reads input byte q (q < n).
using ppi::SYM_LAST;
using ppi::SYM_MID;

__device__ __forceinline__ uint32_t sym_group(const ParseParams& P, const uint8_t* b2g,
                                              uint32_t cp) {
  if (cp < 0x80) return b2g[cp];
  for (uint32_t k = 0; k < P.sym_n; ++k)
    if (P.sym_cp[k] == cp) return P.sym_g[k];
  return P.sym_dflt;
}
__device__ __forceinline__ bool is_cont(uint32_t b) { return (b & 0xC0u) == 0x80u; }

// UTF-8: the group of the symbol whose last byte is r.
template <class ByteAt>
__device__ uint32_t utf8_group(const ParseParams& P, const uint8_t* b2g, uint64_t r, ByteAt B) {
  uint64_t q = r;
  for (int k = 0; k < 4 && q > 0 && is_cont(B(q)); ++k) --q;
  const uint32_t lead = B(q);
  if (is_cont(lead)) return P.sym_dflt;  // no first byte in reach (or at the input start)
  const uint32_t len = uint32_t(r - q) + 1;
  uint32_t want, v;
  if (lead < 0x80) { want = 1; v = lead; }
  else if ((lead & 0xE0u) == 0xC0u) { want = 2; v = lead & 0x1Fu; }
  else if ((lead & 0xF0u) == 0xE0u) { want = 3; v = lead & 0x0Fu; }
  else if ((lead & 0xF8u) == 0xF0u) { want = 4; v = lead & 0x07u; }
  else return P.sym_dflt;
  if (len != want) return P.sym_dflt;
  for (uint64_t i = q + 1; i <= r; ++i) v = (v << 6) | (B(i) & 0x3Fu);
  const uint32_t lo = len == 2 ? 0x80u : len == 3 ? 0x800u : len == 4 ? 0x10000u : 0u;
  if (v < lo || v > 0x10FFFFu) return P.sym_dflt;
  return sym_group(P, b2g, v);
}

// The code of input byte p.
template <class ByteAt>
__device__ uint32_t sym_code(const ParseParams& P, const uint8_t* b2g, uint64_t p, ByteAt B) {
  const uint64_t n = P.n;
  if (P.enc == PP_ENC_UTF8) {
    const uint32_t b = B(p);
    if (!(p + 1 < n && is_cont(B(p + 1))))  // the symbol's last byte
      return b < 0x80 ? b : SYM_LAST + utf8_group(P, b2g, p, B);
    uint64_t r = p + 1;  // its last byte, when at most four bytes on
    for (int k = 1; k < 4 && r + 1 < n && is_cont(B(r + 1)); ++k) ++r;
    const bool longer = r + 1 < n && is_cont(B(r + 1));
    return SYM_MID + (longer ? uint32_t(P.sym_dflt) : utf8_group(P, b2g, r, B));
  }
  // UTF-16LE
  const uint64_t u = p >> 1;
  if (2 * u + 1 >= n) return SYM_LAST + P.sym_dflt;  // an odd last byte
  auto unit = [&](uint64_t v) { return B(2 * v) | (B(2 * v + 1) << 8); };
  const uint32_t x = unit(u);
  uint64_t last = 2 * u + 1;
  uint32_t cp = x;
  if (x >= 0xDC00u && x <= 0xDFFFu && u > 0) {
    const uint32_t y = unit(u - 1);
    if (y >= 0xD800u && y <= 0xDBFFu) cp = 0x10000u + ((y - 0xD800u) << 10) + (x - 0xDC00u);
  } else if (x >= 0xD800u && x <= 0xDBFFu && 2 * u + 3 < n) {
    const uint32_t y = unit(u + 1);
    if (y >= 0xDC00u && y <= 0xDFFFu) {
      cp = 0x10000u + ((x - 0xD800u) << 10) + (y - 0xDC00u);
      last = 2 * u + 3;
    }
  }
  if (p == last) return cp < 0x80 ? cp : SYM_LAST + sym_group(P, b2g, cp);
  return SYM_MID + sym_group(P, b2g, cp);
}

// The code of input byte p, read from HBM (the paths outside the tile pass's
// hot loops).
__device__ __noinline__ uint32_t sym_code_global(const ParseParams& P, uint64_t p) {
  auto B = [&](uint64_t q) -> uint32_t { return __ldg(P.in + q); };
  return sym_code(P, P.sym_b2g, p, B);
}

// Symbol codes of tile bytes [c0, c0 + clen) into codes_s[c0 ...]; bytes
// outside the tile (a symbol crossing the tile's ends) are read from HBM.
__device__ __noinline__ void chunk_codes(const ParseParams& P, const uint8_t* b2g,
                                         const uint8_t* tile_s, uint64_t tile_base,
                                         uint32_t tile_len, uint32_t c0, uint32_t clen,
                                         uint8_t* codes_s) {
  auto B = [&](uint64_t q) -> uint32_t {
    const uint64_t l = q - tile_base;
    return l < tile_len ? uint32_t(tile_s[l]) : uint32_t(__ldg(P.in + q));
  };
  for (uint32_t j = 0; j < clen; ++j)
    codes_s[c0 + j] = uint8_t(sym_code(P, b2g, tile_base + c0 + j, B));
}

// ------------------------------------------------- tile feeding (TMA)
// Two linear landing buffers.  A block takes its first tile at start; once
// a tile has landed it takes the next ticket and starts that tile's bulk
// copy into the other buffer, which the previous tile released at its last
// block barrier, so the copy runs while the current tile is processed.
// Neither pass waits on another tile, so the order in which tickets are
// taken carries no constraint.
struct Feed {
  uint64_t bar[2];
  uint32_t tile[2], issued[2], parity[2];
  uint32_t cur;
};

__device__ __forceinline__ uint32_t issue_tile(const ParseParams& P, uint32_t tile, bool aligned_in,
                                               uint8_t* lin_s, uint64_t* bar) {
  if (tile >= P.n_tiles || !aligned_in) return 0;
  const uint64_t tb = uint64_t(tile) * TILE;
  const uint32_t bytes = uint32_t(min(uint64_t(TILE), P.n - tb)) & ~15u;
  if (!bytes) return 0;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(lin_s, P.in + tb, bytes, bar);
  return 1;
}

// tk (thread 0 only) holds the ticket of the tile after the current one:
// each ticket is taken one tile before it is used, so the atomic's round
// trip never stalls the block.
__device__ __forceinline__ void feed_start(const ParseParams& P, Feed& F, uint32_t* counter,
                                           bool aligned_in, uint8_t* lin0, uint32_t& tk) {
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&F.bar[b], 1);
      F.parity[b] = 0;
      F.issued[b] = 0;
    }
    F.tile[0] = atomicAdd(counter, 1u);
    F.issued[0] = issue_tile(P, F.tile[0], aligned_in, lin0, &F.bar[0]);
    F.cur = 0;
    tk = atomicAdd(counter, 1u);
  }
  __syncthreads();
}

// Wait until the current tile is in its landing buffer (plain loads for a
// ragged tail or unaligned input), take the next ticket and start that
// tile's copy into the other buffer, and load this thread's chunk words.
__device__ __forceinline__ void feed_tile(const ParseParams& P, Feed& F, uint32_t* counter,
                                          bool aligned_in, uint8_t* lin0, uint64_t tile_base,
                                          uint32_t tile_len, uint32_t (&w)[8], uint32_t& tk) {
  const int t = threadIdx.x;
  const uint32_t b = F.cur;
  uint8_t* lin_s = lin0 + b * TILE;
  const uint32_t bulk = F.issued[b] ? (tile_len & ~15u) : 0u;
  if (F.issued[b]) {
    if (!mbar_wait_bounded(&F.bar[b], F.parity[b], WAIT_LIMIT)) {
      if (t == 0) report(P.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
      mbar_wait_bounded(&F.bar[b], F.parity[b], WAIT_LIMIT);
    }
  }
  if (bulk < tile_len) {
    for (uint32_t k = bulk + t; k < tile_len; k += NT) lin_s[k] = P.in[tile_base + k];
    __syncthreads();
  }
  if (t == 0) {
    const uint32_t o = b ^ 1u;
    F.tile[o] = tk;
    F.issued[o] = issue_tile(P, tk, aligned_in, lin0 + o * TILE, &F.bar[o]);
    tk = atomicAdd(counter, 1u);
  }
  const uint4* src = reinterpret_cast<const uint4*>(lin_s + uint32_t(t) * CB);
  const int sw = (t >> 2) & 1;  // alternate read order: conflict-free 16-byte reads
  const uint4 x = src[sw], y = src[sw ^ 1];
  const uint4 lo = sw ? y : x, hi = sw ? x : y;
  w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
  w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
}

// After the last read of the current buffer (the caller's earlier block
// barrier): switch to the other buffer, whose tile is already on its way.
__device__ __forceinline__ void feed_next(Feed& F) {
  if (threadIdx.x == 0) {
    const uint32_t b = F.cur;
    if (F.issued[b]) F.parity[b] ^= 1u;
    F.cur = b ^ 1u;
  }
  __syncthreads();
}

__device__ __forceinline__ void feed_finish(Feed& F) {
  // never leave with a bulk copy in flight into this CTA's shared memory
  // (only the current buffer can have one: a copy is started only for a
  // tile that exists, and every such tile is processed, so waited for,
  // before the loop ends)
  if (threadIdx.x == 0 && F.issued[F.cur]) mbar_wait_bounded(&F.bar[F.cur], F.parity[F.cur], WAIT_LIMIT);
}

// Multi-instance DFA over the chunk (back to front): G := G o delta_group(b).
// Also returns the chunk's non-background bytes (special) and the bytes that
// are not inert in the sticky state (special_x).
__device__ __forceinline__ void stv_pass(const uint32_t (&w)[8], uint32_t clen, const uint8_t* tile_s,
                                         uint32_t cstart, const uint32_t* my_lut, uint32_t& G,
                                         uint32_t& special, uint32_t& special_x) {
  G = STV_ID;
  special = 0;
  special_x = 0;
  if (clen == CB) {
#pragma unroll
    for (int j = CB - 1; j >= 0; --j) {
      const uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      const uint32_t e = my_lut[b << 5];
      G = __byte_perm(G, STV_INV_POOL, e);
      special = __funnelshift_l(e, special, 1);
      special_x = __funnelshift_l(e << 1, special_x, 1);
    }
  } else {
    for (int j = int(clen) - 1; j >= 0; --j) {
      const uint32_t e = my_lut[tile_byte(tile_s, cstart + j) << 5];
      G = __byte_perm(G, STV_INV_POOL, e);
      special = __funnelshift_l(e, special, 1);
      special_x = __funnelshift_l(e << 1, special_x, 1);
    }
  }
}

// Compose chunk vectors across the block.  Returns the thread's exclusive
// vector inside the warp; warp exclusive vectors go to warp_stv[], the tile
// aggregate to *tile_stv.
__device__ __forceinline__ uint32_t block_stv(uint32_t G, uint32_t* warp_stv, uint32_t* tile_stv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = G;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, inc, d);
    if (lane >= d) inc = stv_compose(o, inc);
  }
  uint32_t lane_ex = __shfl_up_sync(FULL, inc, 1);
  if (lane == 0) lane_ex = STV_ID;
  if (lane == 31) warp_stv[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = lane < NW ? warp_stv[lane] : STV_ID;
    uint32_t wi = v;
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, wi, d);
      if (lane >= d) wi = stv_compose(o, wi);
    }
    uint32_t wex = __shfl_up_sync(FULL, wi, 1);
    if (lane == 0) wex = STV_ID;
    if (lane < NW) warp_stv[lane] = wex;
    if (lane == NW - 1) *tile_stv = wi;
  }
  __syncthreads();
  return lane_ex;
}

// Re-run one DFA from state s over the chunk's non-background bytes: the
// three bitmap indexes (ParPaRaw Section 3.1) plus the first invalid byte,
// the last terminator ((tile pos + 1) << 8 | state after) and the end state.
struct Tags { uint32_t fd, rd, ctrl, inv_at, last, end; };

__device__ __forceinline__ Tags tag_chunk(uint32_t s, uint32_t special, uint32_t special_x,
                                          uint32_t sticky, uint32_t clen, uint32_t cstart,
                                          const uint8_t* own, const uint32_t* my_lut,
                                          uint32_t bg_next) {
  Tags r = {0u, 0u, 0u, 32u, 0u, s};
  if (s == 4) { r.inv_at = 0; return r; }
  uint32_t m = special & range_mask(0, clen);
  uint32_t prev = 0;
  if (s == sticky) {  // bytes inert in the sticky state leave it and tag DATA
    const uint32_t mx = special_x & range_mask(0, clen);
    if (!mx) return r;
    prev = __ffs(mx) - 1;
    m &= ~range_mask(0, prev);
  }
  while (m) {
    const uint32_t j = __ffs(m) - 1;
    m &= m - 1;
    if (j > prev) {  // a run of background bytes: one idempotent transition
      const uint32_t s1 = (bg_next >> (4 * s)) & 0xFu;
      if (s1 == 4) { r.inv_at = prev; r.end = 4; return r; }
      s = s1;
    }
    const uint32_t byte = own[j];
    const uint32_t e = my_lut[byte << 5];
    const uint32_t nx = (e >> (4 * s)) & 0xFu;
    if (nx == 4) { r.inv_at = j; r.end = 4; return r; }
    const uint32_t tg = (e >> (20 + 2 * s)) & 3u;
    const uint32_t bit = 1u << j;
    r.fd |= tg == PP_TAG_FD ? bit : 0u;
    r.rd |= tg == PP_TAG_RD ? bit : 0u;
    r.ctrl |= tg == PP_TAG_CTRL ? bit : 0u;
    if (tg == PP_TAG_FD || tg == PP_TAG_RD) r.last = ((cstart + j + 1) << 8) | nx;
    s = nx;
    prev = j + 1;
  }
  if (prev < clen) {
    const uint32_t s1 = (bg_next >> (4 * s)) & 0xFu;
    if (s1 == 4) { r.inv_at = prev; r.end = 4; return r; }
    s = s1;
  }
  r.end = s;
  return r;
}

__device__ __forceinline__ V2 chunk_v2(const Tags& g) {
  V2 v;
  v.rec = __popc(g.rd);
  if (g.rd) {
    const uint32_t hi = 31 - __clz(g.rd);
    v.col = ABS32 | uint32_t(__popc(hi == 31 ? 0u : (g.fd >> (hi + 1))));
  } else {
    v.col = uint32_t(__popc(g.fd));
  }
  v.last = g.last;
  return v;
}

// Feed the value bytes of field [fs, fe) (global offsets) to a numeric
// accumulator; returns the number of value bytes.  A field inside the tile
// reads the tile copy (skipping control bytes by the control bitmap); a
// field that began in an earlier tile is re-read from global memory and
// re-tagged by running the DFA from the state at its first byte (lut: one
// LUT entry per byte value).
template <class Acc>
__device__ __forceinline__ uint32_t feed_field(Acc& acc, const ParseParams& P, uint64_t fs,
                                               uint64_t fe, uint64_t tile_base,
                                               const uint8_t* tile_s, const uint32_t* ctrl_s,
                                               const uint32_t* lut, uint32_t fstate) {
  uint32_t ndata = 0;
  if (fs >= tile_base) {
    const uint32_t a = uint32_t(fs - tile_base), e = uint32_t(fe - tile_base);
    if (popc_range(ctrl_s, a, e) == 0) {
      for (uint32_t p = a; p < e; ++p) acc.feed(tile_byte(tile_s, p));
      ndata = e - a;
    } else {
      for (uint32_t p = a; p < e; ++p) {
        if ((ctrl_s[p >> 5] >> (p & 31)) & 1u) continue;
        acc.feed(tile_byte(tile_s, p));
        ++ndata;
      }
    }
  } else {
    uint32_t s = fstate;
    for (uint64_t p = fs; p < fe; ++p) {
      const uint32_t b = p >= tile_base ? tile_byte(tile_s, uint32_t(p - tile_base))
                                        : uint32_t(__ldg(P.in + p));
      const uint32_t e = lut[b];  // byte inputs only: with an encoding such fields go to a warp
      const uint32_t tg = (e >> (20 + 2 * s)) & 3u;
      s = (e >> (4 * s)) & 0xFu;
      if (tg == uint32_t(PP_TAG_CTRL)) continue;
      acc.feed(b);
      ++ndata;
    }
  }
  return ndata;
}

// ---------------------------------------------- word access to the tile
__device__ __forceinline__ uint32_t tile_word(const uint32_t* tile_w, uint32_t q) { return tile_w[q]; }
// 8 bytes of a buffer from byte position p (little-endian: byte p lowest);
// bytes past the tile are unspecified but stay inside shared memory.
__device__ __forceinline__ uint64_t tile_load8(const uint32_t* tile_w, uint32_t p) {
  const uint32_t q = p >> 2, sh = (p & 3u) * 8u;
  const uint32_t w0 = tile_word(tile_w, q), w1 = tile_word(tile_w, q + 1),
                 w2 = tile_word(tile_w, q + 2);
  return uint64_t(__funnelshift_r(w0, w1, sh)) | (uint64_t(__funnelshift_r(w1, w2, sh)) << 32);
}

__device__ __forceinline__ void load_lut(const ParseParams& P, uint32_t* lut_s) {
  for (int k = threadIdx.x; k < 256 * 32; k += NT) lut_s[k] = P.lut[k >> 5];
}

// ======================================================= 0. tile start states
// The context pass works from each tile's true start state, found first by a
// transition-vector pass (ParPaRaw Section 3.1) and an exclusive composite
// scan over tiles.
constexpr int TV_NT = 256;              // tile-vector pass: a warp per tile
constexpr int TV_BYTES = TILE / 32;     // bytes per lane
constexpr int TV_STEP = 128;            // staged path: bytes per lane per step
constexpr int TV_ROW = TV_STEP + 16;    // a lane's staging row (padded: conflict-free reads)
constexpr int TV_SMEM = LUT_BYTES + (TV_NT / 32) * 32 * TV_ROW;
constexpr int TS_NT = 256, TS_TPT = 16; // tile-state scan: tiles per thread
constexpr int TS_TILES = TS_NT * TS_TPT;

// Transition vector of each tile: one warp per tile, each lane folding
// TV_BYTES bytes back to front, a warp scan composing the lanes in order.
// A whole tile of a 16-byte aligned byte input goes through shared memory
// in steps of TV_STEP bytes per lane: a lane's bytes are TV_BYTES from its
// neighbour's, so reading them straight from global memory would touch a
// sector per lane in every load; the warp instead loads the step's rows
// 128 contiguous bytes per 8 lanes, stores them to per-lane rows padded to
// TV_ROW bytes, and each lane folds its own row.  Launched with TV_SMEM
// bytes of dynamic shared memory.
__global__ void __launch_bounds__(TV_NT) tile_stv_kernel(const __grid_constant__ ParseParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint8_t b2g_s[0x80];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* const stage = smem + LUT_BYTES + (threadIdx.x >> 5) * (32 * TV_ROW);  // the warp's rows
  for (int k = threadIdx.x; k < 256 * 32; k += TV_NT) lut_s[k] = P.lut[k >> 5];
  for (int k = threadIdx.x; k < 0x80; k += TV_NT) b2g_s[k] = P.sym_b2g[k];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint32_t* my_lut = lut_s + lane;
  // A lane's bytes split into a head up to the first 16-byte boundary, whole
  // 16-byte blocks and a tail; with the input 16-byte aligned there is no
  // head or tail.  The split is the same for every lane (lanes start at
  // multiples of TV_BYTES).
  const uint32_t h = uint32_t(16u - (reinterpret_cast<uintptr_t>(P.in) & 15u)) & 15u;
  const uint32_t nb = (TV_BYTES - h) >> 4;          // TV_BYTES / 16, or one less
  const uint32_t tl = TV_BYTES - h - 16u * nb;      // 0, or 16 - h
  const uint32_t warps = gridDim.x * (TV_NT / 32);
  auto fold16 = [&](uint32_t G, const uint4 v) {
    const uint32_t wq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 15; j >= 0; --j)
      G = __byte_perm(G, STV_INV_POOL, my_lut[((wq[j >> 2] >> (8 * (j & 3))) & 0xFFu) << 5]);
    return G;
  };
  for (uint32_t tile = blockIdx.x * (TV_NT / 32) + (threadIdx.x >> 5); tile < P.n_tiles;
       tile += warps) {
    const uint64_t b0 = uint64_t(tile) * TILE + uint64_t(lane) * TV_BYTES;
    const uint32_t len = b0 < P.n ? uint32_t(min(uint64_t(TV_BYTES), P.n - b0)) : 0u;
    uint32_t G = STV_ID;
    if (P.enc) {
      // Symbols of an encoding: only a symbol's last byte moves the state
      // (its other bytes have identity rows), so only last bytes are
      // decoded.  UTF-8 blocks of 16 bytes below 0x80, not followed by a
      // continuation byte, are their own codes and fold like bytes.
      auto B = [&](uint64_t q) -> uint32_t { return __ldg(P.in + q); };
      auto fold_sym = [&](uint32_t G, uint64_t p) {
        if (P.enc == PP_ENC_UTF8 ? (p + 1 < P.n && is_cont(B(p + 1)))
                                 : ((p & 1u) == 0 && p + 1 < P.n))
          return G;  // not the symbol's last byte
        return __byte_perm(G, STV_INV_POOL, my_lut[sym_code(P, b2g_s, p, B) << 5]);
      };
      const bool vec = P.enc == PP_ENC_UTF8 && len == TV_BYTES &&
                       (reinterpret_cast<uintptr_t>(P.in + b0) & 15u) == 0;
      if (vec) {
        const uint4* src = reinterpret_cast<const uint4*>(P.in + b0);
        uint32_t next = b0 + TV_BYTES < P.n ? B(b0 + TV_BYTES) : 0u;  // the byte after the block
        for (int k = TV_BYTES / 16 - 1; k >= 0; --k) {
          const uint4 v = __ldg(src + k);
          if ((((v.x | v.y | v.z | v.w) & 0x80808080u) == 0) && !is_cont(next)) {
            G = fold16(G, v);
          } else {
            for (int j = 15; j >= 0; --j) G = fold_sym(G, b0 + 16u * uint32_t(k) + uint32_t(j));
          }
          next = v.x & 0xFFu;
        }
      } else {
        for (int j = int(len) - 1; j >= 0; --j) G = fold_sym(G, b0 + uint32_t(j));
      }
    } else if (h == 0 && uint64_t(tile + 1) * TILE <= P.n) {  // staged (uniform in the warp)
      const uint8_t* tb = P.in + uint64_t(tile) * TILE;
      const uint32_t r4 = uint32_t(lane) >> 3, c16 = uint32_t(lane) & 7u;
      for (int st = TV_BYTES / TV_STEP - 1; st >= 0; --st) {
        __syncwarp();  // the rows of the step after are read
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t row = 4u * uint32_t(q) + r4;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(tb + row * TV_BYTES + uint32_t(st) * TV_STEP) + c16);
          *reinterpret_cast<uint4*>(stage + row * TV_ROW + c16 * 16u) = v;
        }
        __syncwarp();
        const uint4* mine = reinterpret_cast<const uint4*>(stage + uint32_t(lane) * TV_ROW);
#pragma unroll
        for (int k = TV_STEP / 16 - 1; k >= 0; --k) G = fold16(G, mine[k]);
      }
    } else if (len == TV_BYTES) {
      const uint8_t* p = P.in + b0;
      for (int j = int(tl) - 1; j >= 0; --j)  // the tail
        G = __byte_perm(G, STV_INV_POOL, my_lut[uint32_t(__ldg(p + h + 16u * nb + j)) << 5]);
      const uint4* src = reinterpret_cast<const uint4*>(p + h);
      const uint32_t ng = nb >> 2;  // groups of four blocks; the rest first, back to front
      for (int k = int(nb) - 1; k >= int(4 * ng); --k) G = fold16(G, __ldg(src + k));
      // groups back to front, the next group's loads in flight while the
      // current one folds
      uint4 cur[4], nxt[4] = {};
#pragma unroll
      for (int k = 0; k < 4; ++k) cur[k] = __ldg(src + 4 * (ng - 1) + k);
      for (int step = int(ng) - 1; step >= 0; --step) {
        if (step > 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) nxt[k] = __ldg(src + 4 * (step - 1) + k);
        }
#pragma unroll
        for (int k = 3; k >= 0; --k) G = fold16(G, cur[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
      }
      for (int j = int(h) - 1; j >= 0; --j)  // the head
        G = __byte_perm(G, STV_INV_POOL, my_lut[uint32_t(__ldg(p + j)) << 5]);
    } else {
      for (int j = int(len) - 1; j >= 0; --j)
        G = __byte_perm(G, STV_INV_POOL, my_lut[uint32_t(__ldg(P.in + b0 + j)) << 5]);
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, G, d);
      if (lane >= d) G = stv_compose(o, G);
    }
    if (lane == 31) P.s.tile_stv[tile] = G;
  }
}

// Exclusive composite scan of the tile vectors (single-pass decoupled
// look-back between blocks, bounded waits), applied to the start state.
__global__ void __launch_bounds__(TS_NT) tile_state_kernel(const __grid_constant__ ParseParams P) {
  __shared__ uint32_t blk_s, wv[TS_NT / 32], pre_s;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) blk_s = atomicAdd(&P.s.counters[3], 1u);
  __syncthreads();
  const uint32_t blk = blk_s;
  const uint32_t t0 = blk * TS_TILES + uint32_t(t) * TS_TPT;
  uint32_t v[TS_TPT];
  uint32_t acc = STV_ID;
#pragma unroll
  for (int e = 0; e < TS_TPT; ++e) {
    v[e] = t0 + e < P.n_tiles ? P.s.tile_stv[t0 + e] : STV_ID;
    acc = stv_compose(acc, v[e]);
  }
  uint32_t inc = acc;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, inc, d);
    if (lane >= d) inc = stv_compose(o, inc);
  }
  uint32_t lex = __shfl_up_sync(FULL, inc, 1);
  if (lane == 0) lex = STV_ID;
  if (lane == 31) wv[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    constexpr int W = TS_NT / 32;
    const uint32_t x0 = lane < W ? wv[lane] : STV_ID;
    uint32_t x = x0;
#pragma unroll
    for (int d = 1; d < W; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, x, d);
      if (lane >= d) x = stv_compose(o, x);
    }
    uint32_t xe = __shfl_up_sync(FULL, x, 1);
    if (lane == 0) xe = STV_ID;
    const uint32_t agg = __shfl_sync(FULL, x, W - 1);
    __syncwarp();
    if (lane < W) wv[lane] = xe;
    const uint32_t pre = lookback_word(P.s.tstate_words, blk, agg, STV_ID, STV_ID,
                                       [](uint32_t a, uint32_t b) { return stv_compose(a, b); },
                                       LookbackCfg{P.st, P.spin_limit});
    if (lane == 0) pre_s = pre;
  }
  __syncthreads();
  uint32_t s = stv_apply(pre_s, P.start_state);
  s = stv_apply(wv[warp], s);
  s = stv_apply(lex, s);
#pragma unroll
  for (int e = 0; e < TS_TPT; ++e)
    if (t0 + e < P.n_tiles) {
      P.s.tile_state[t0 + e] = uint8_t(s);
      s = stv_apply(v[e], s);
    }
}

// Numeric field whose bytes are not all in the tile, contain control bytes
// or need the full grammar: streaming accumulators over the value bytes.
// Returns the error bits; *out receives the value (dflt, the column's
// default, for a field without value bytes; 0 after an error).
__device__ __forceinline__ int convert_general(const ParseParams& P, uint32_t ty, uint64_t fs,
                                            uint64_t fe, uint64_t tile_base,
                                            const uint8_t* tile_s, const uint32_t* ctrl_s,
                                            const uint32_t* my_lut, uint32_t fstate,
                                            uint64_t dflt, uint64_t* out) {
  int err = 0;
  uint64_t val = dflt;
  if (ty == PP_COL_FLOAT64) {
    ppn::FloatAcc acc;
    const uint32_t nd = feed_field(acc, P, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
    if (nd) err = acc.finish(&val);
  } else if (ty == PP_COL_TIMESTAMP) {
    ppn::TsAcc acc;
    const uint32_t nd = feed_field(acc, P, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
    if (nd) {
      int64_t x = 0;
      err = acc.finish(&x);
      val = uint64_t(x);
    }
  } else {
    ppn::IntAcc acc;
    const uint32_t nd = feed_field(acc, P, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
    if (nd) {
      int64_t x = 0;
      if (ty == PP_COL_INT8) err = acc.finish(128ull, 127ull, &x);
      else if (ty == PP_COL_INT32) err = acc.finish(2147483648ull, 2147483647ull, &x);
      else err = acc.finish(9223372036854775808ull, 9223372036854775807ull, &x);
      val = uint64_t(x);
    }
  }
  *out = val;
  return err;
}

// The tile context a numeric field's conversion needs.
struct NumCtx {
  uint64_t tile_base, tile_fstart;  // the tile's first byte; start of the field open at it
  uint32_t tile_fstate;             // DFA state at tile_fstart
  const uint8_t* tile_s;            // tile byte p at tile_s[p]
  const uint32_t* raw_w;            // landing buffer as words: tile byte p at byte p + toff
  uint32_t toff;
  const uint32_t* ctrl_s;           // control bitmap per chunk
  const uint32_t* wc;               // control bytes before each warp's chunks ([16]: total)
  const uint16_t* cpl;              // control bytes before each chunk inside its warp
  const uint32_t* lut;               // one LUT entry per byte value
  bool any_ctrl;
};

// control bytes of the tile before position p (p <= tile length)
__device__ __forceinline__ uint32_t ctrl_x(const NumCtx& X, uint32_t p) {
  const uint32_t c = p >> 5, b = p & 31u;
  return X.wc[c >> 5] + X.cpl[c] + (b ? uint32_t(__popc(X.ctrl_s[c] & ((1u << b) - 1u))) : 0u);
}

// Convert the numeric field in slot value v (tile-relative start << 16 |
// end; start 0xFFFF = the field began in an earlier tile; SLOT_DEFAULT = a
// missing field) for a column of type TY.  A plain field inside the tile
// and free of control bytes is decoded word-parallel: at most 8 characters
// after the sign (an integer, or for floats a decimal with one '.'
// converted by short_decimal_to_binary64), an integer of 9 to 16 digits
// in two such words, or a timestamp from five words.  Everything else
// streams through the accumulators.
// Returns the error bits; val gets the value's bits (0 for an empty field
// or an error).
template <int TY>
__device__ __forceinline__ int convert_field(const ParseParams& P, uint32_t v, const NumCtx& X,
                                             uint64_t dflt, uint64_t& val) {
  val = 0;
  if (v == SLOT_DEFAULT) { val = dflt; return 0; }  // a missing field: the column default
  const uint32_t fsr = v >> 16, fe = v & 0xFFFFu;
  if (fsr != 0xFFFFu &&
      (!X.any_ctrl || ctrl_x(X, fe) == ctrl_x(X, fsr))) {
    const uint32_t L = fe - fsr;
    if (L == 0) { val = dflt; return 0; }  // an empty field: the column default
    if (TY == PP_COL_TIMESTAMP) {  // five words of the tile from the field start
      const uint32_t a = fsr + X.toff, q = a >> 2, sh = (a & 3u) * 8u;
      uint32_t x[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) x[k] = __funnelshift_r(X.raw_w[q + k], X.raw_w[q + k + 1], sh);
      int64_t t = 0;
      const int err = ppn::parse_timestamp(x, L, &t);
      val = uint64_t(t);
      return err;
    }
    const uint32_t c0 = X.tile_s[fsr];
    const uint32_t sg = (c0 == '-' || c0 == '+') ? 1u : 0u;
    const bool neg = c0 == '-';
    const int n = int(L - sg);
    const uint32_t pv = fsr + sg + X.toff, q = pv >> 2, sh = (pv & 3u) * 8u;
    const uint32_t w0 = X.raw_w[q], w1 = X.raw_w[q + 1];
    const uint32_t x0 = __funnelshift_r(w0, w1, sh);
    uint32_t w;
    if (TY != PP_COL_FLOAT64 && n >= 1 && n <= 4) {  // up to 4 digits: one word
      const uint32_t y = x0 ^ 0x30303030u, a = 32u - 8u * uint32_t(n);
      if (!(ppn::nondigit_bytes(y) & (0x80808080u >> a))) {
        w = ppn::val4(y << a);
        if (TY == PP_COL_INT8 && w > (neg ? 128u : 127u)) return PP_ERR_NUM_OVERFLOW;
        val = neg ? uint64_t(0) - w : uint64_t(w);
        return 0;
      }
    }
    const uint32_t x1 = __funnelshift_r(w1, X.raw_w[q + 2], sh);
    const uint64_t x = (uint64_t(x1) << 32) | x0;
    int k;
    if (n >= 1 && n <= 8 &&
        ppn::short_decimal(uint32_t(x), uint32_t(x >> 32), n, TY == PP_COL_FLOAT64, &w, &k)) {
      if (TY == PP_COL_FLOAT64) {
        val = (w ? ppn::short_decimal_to_binary64(w, k) : 0ull) | (neg ? (1ull << 63) : 0ull);
        return 0;
      }
      if (TY == PP_COL_INT8 && w > (neg ? 128u : 127u)) return PP_ERR_NUM_OVERFLOW;
      val = neg ? uint64_t(0) - w : uint64_t(w);
      return 0;
    }
    if (TY != PP_COL_FLOAT64 && n > 8 && n <= 16) {
      const uint64_t x2 = tile_load8(X.raw_w, fsr + sg + 8 + X.toff);
      uint32_t wl;
      if (ppn::short_decimal(uint32_t(x), uint32_t(x >> 32), 8, false, &w, &k) &&
          ppn::short_decimal(uint32_t(x2), uint32_t(x2 >> 32), n - 8, false, &wl, &k)) {
        uint32_t p10 = 10u;  // 10^(n - 8)
        for (int i = 9; i < n; ++i) p10 *= 10u;
        const uint64_t mag = uint64_t(w) * p10 + wl;
        const uint64_t lim = TY == PP_COL_INT8 ? 127ull : TY == PP_COL_INT32 ? 2147483647ull
                                                                              : 9223372036854775807ull;
        if (mag > lim + (neg ? 1u : 0u)) return PP_ERR_NUM_OVERFLOW;
        val = neg ? ~mag + 1 : mag;
        return 0;
      }
    }
  }
  return convert_general(P, TY, fsr == 0xFFFFu ? X.tile_fstart : X.tile_base + fsr,
                         X.tile_base + fe, X.tile_base, X.tile_s, X.ctrl_s, X.lut,
                         X.tile_fstate, dflt, &val);
}

// Convert one row's field (slot value v) of a column of type TY, store it
// at out[rec] and report a number error at the field's first byte.
template <int TY>
__device__ __forceinline__ void convert_store(const ParseParams& P, const NumCtx& X, void* out,
                                              uint64_t rec, uint32_t v, uint64_t dflt) {
  uint64_t val;
  const int err = convert_field<TY>(P, v, X, dflt, val);
  if (TY == PP_COL_INT32) static_cast<int32_t*>(out)[rec] = int32_t(val);
  else if (TY == PP_COL_INT8) static_cast<int8_t*>(out)[rec] = int8_t(val);
  else static_cast<uint64_t*>(out)[rec] = val;
  if (err) {
    const uint32_t fsr = v >> 16;
    report(P.st, err, fsr == 0xFFFFu ? X.tile_fstart : X.tile_base + fsr, true);
  }
}

// ------------------------------------------- long numeric fields (a warp)
// Collaboration on long fields (ParPaRaw Section 3.3): a number field whose
// bytes span more than LONG_NUM bytes is not converted by its lane in the
// tile pass.  The lane queues it (up to LONG_CAP fields per call; fields
// beyond that are converted by their lane), and long_field_kernel converts
// each queued field with a whole warp, by the data-parallel method of the
// parse itself:
//  1. the warp takes the bytes from the start of the field's tile, whose DFA
//     state the tile-state scan gave, to the field's end, in rounds of
//     32 x LONG_SEG bytes, a segment per lane; a warp scan of the segments'
//     transition vectors gives each segment its CSV state (Section 3.1), and
//     with it which of its bytes are control bytes;
//  2. the field's value bytes run through the number grammar as a second DFA
//     (9 states), again by transition vectors and a warp scan, which gives
//     each segment its grammar state; each lane then counts its integer- and
//     fraction-part digits and finds its first non-zero digits;
//  3. warp sums and minima combine the segments and rounds, and one lane
//     reads at most 19 significant digits (and at most 7 of the exponent)
//     and finishes the conversion.
// The value is the one the per-lane conversion gives (the first 19
// significant digits, the exponent saturated the same way).
constexpr uint32_t LONG_NUM = 256;
constexpr uint32_t LONG_SEG = 16;
constexpr int LF_NT = 128;

namespace numg {
// Number grammar [+-]?([0-9]+(\.[0-9]*)?|\.[0-9]+)([eE][+-]?[0-9]+)?:
// G0 start, G1 after the sign, G2 integer digits, G3 a point with no digit
// before, G4 fraction (after at least one mantissa digit), G5 after the
// exponent mark, G6 after its sign, G7 exponent digits, GX error.  Accepting:
// G2, G4, G7 (integers: G2 alone).  Symbol classes: digit, sign, point,
// exponent mark, other.  A vector holds the next state of every state, one
// nibble per state (states 9-15 unused, mapped to themselves).
constexpr uint32_t G0 = 0, G1 = 1, G2 = 2, G3 = 3, G4 = 4, G5 = 5, G6 = 6, G7 = 7, GX = 8;
constexpr uint64_t vec9(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                        uint32_t a5, uint32_t a6, uint32_t a7) {
  const uint32_t a[9] = {a0, a1, a2, a3, a4, a5, a6, a7, GX};
  uint64_t v = 0;
  for (int s = 0; s < 16; ++s) v |= uint64_t(s < 9 ? a[s] : uint32_t(s)) << (4 * s);
  return v;
}
constexpr uint64_t K_DIGIT = vec9(G2, G2, G2, G4, G4, G7, G7, G7);
constexpr uint64_t K_SIGN = vec9(G1, GX, GX, GX, GX, G6, GX, GX);
constexpr uint64_t K_POINT = vec9(G3, G3, G4, GX, GX, GX, GX, GX);
constexpr uint64_t K_EXP = vec9(GX, GX, G5, GX, G5, GX, GX, GX);
constexpr uint64_t K_OTHER = vec9(GX, GX, GX, GX, GX, GX, GX, GX);
__device__ __forceinline__ uint32_t sym_class(uint32_t b) {
  return b - '0' <= 9u ? 0u : (b == '+' || b == '-') ? 1u : b == '.' ? 2u
                                                      : (b | 0x20u) == 'e' ? 3u : 4u;
}
__device__ __forceinline__ uint64_t class_vec(uint32_t c) {
  return c == 0 ? K_DIGIT : c == 1 ? K_SIGN : c == 2 ? K_POINT : c == 3 ? K_EXP : K_OTHER;
}
}  // namespace numg

// Byte b, whose DFA state before it is s, is a control byte; s advances past it.
__device__ __forceinline__ bool step_ctrl(const uint32_t* lut, uint32_t b, uint32_t& s) {
  const uint32_t e = lut[b];
  const uint32_t tg = (e >> (20 + 2 * s)) & 3u;
  s = (e >> (4 * s)) & 0xFu;
  return tg == uint32_t(PP_TAG_CTRL);
}
__device__ __forceinline__ uint64_t warp_min64(uint64_t v) {
#pragma unroll
  for (int d = 16; d; d >>= 1) v = min(v, __shfl_xor_sync(FULL, v, d));
  return v;
}

// Convert queued field f with the calling warp; lane 0 stores the value and
// reports an error at the field's first byte.  lut: one entry per byte value.
__device__ void convert_long(const ParseParams& P, const uint32_t* lut, const ppi::LongField f) {
  using namespace numg;
  constexpr uint64_t NONE = ~0ull;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t ty = f.col >> 8, col = f.col & 0xFFu;
  const uint64_t gs = f.start, ge = f.end;
  auto code_at = [&](uint64_t q, uint32_t b) -> uint32_t {  // the LUT index of byte q (value b)
    return P.enc ? sym_code_global(P, q) : b;
  };
  // where the walk starts: the field's start when its DFA state is known,
  // else the start of its tile (whose state the tile-state scan gave)
  const bool known = (f.state & ppi::LONG_STATE) != 0;
  const uint64_t t0 = known ? gs : (gs / TILE) * TILE;
  uint32_t cs = known ? (f.state & 0xFFu) : P.s.tile_state[gs / TILE];  // CSV state at the round start
  uint32_t gq = G0;                         // grammar state at the round start
  uint64_t n_int = 0, n_frac = 0, n_val = 0;
  uint64_t z = NONE, pz = NONE, pez = NONE;  // first non-zero mantissa digit (index, position), exponent digit
  uint32_t sz = 0, sez = 0;                   // CSV states before them
  bool mneg = false, eneg = false;
  for (uint64_t r0 = t0; r0 < ge; r0 += 32 * LONG_SEG) {
    const uint64_t a = r0 + uint64_t(lane) * LONG_SEG;
    const uint32_t len = a < ge ? uint32_t(min(uint64_t(LONG_SEG), ge - a)) : 0u;
    uint32_t bw[LONG_SEG / 4] = {};  // the segment's bytes, four to a word
#pragma unroll
    for (uint32_t j = 0; j < LONG_SEG; ++j)
      if (j < len) bw[j >> 2] |= uint32_t(__ldg(P.in + a + j)) << (8 * (j & 3));
    // CSV states: a warp scan of the segments' transition vectors
    uint32_t cv = STV_ID;
#pragma unroll
    for (int j = int(LONG_SEG) - 1; j >= 0; --j)
      if (uint32_t(j) < len) cv = __byte_perm(cv, STV_INV_POOL, lut[code_at(a + j, (bw[j >> 2] >> (8 * (j & 3))) & 0xFFu)]);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, cv, d);
      if (int(lane) >= d) cv = stv_compose(o, cv);
    }
    uint32_t cx = __shfl_up_sync(FULL, cv, 1);
    if (lane == 0) cx = STV_ID;
    const uint32_t s_lane = stv_apply(cx, cs);
    cs = stv_apply(__shfl_sync(FULL, cv, 31), cs);
    uint32_t val_m = 0;  // bit j: byte j is a value byte of the field
    {
      uint32_t s = s_lane;
#pragma unroll
      for (uint32_t j = 0; j < LONG_SEG; ++j)
        if (j < len && !step_ctrl(lut, code_at(a + j, (bw[j >> 2] >> (8 * (j & 3))) & 0xFFu), s) &&
            a + j >= gs)
          val_m |= 1u << j;
    }
    // grammar: the segment's transition vector (runs of digits compose once)
    Stv16 gv = stv16_id();
    {
      uint32_t last = 5;
#pragma unroll
      for (uint32_t j = 0; j < LONG_SEG; ++j) {
        if (!((val_m >> j) & 1u)) continue;
        const uint32_t c = sym_class((bw[j >> 2] >> (8 * (j & 3))) & 0xFFu);
        if (!(c == 0 && last == 0)) gv = stv16_compose(gv, stv16_unpack(class_vec(c)));
        last = c;
      }
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const Stv16 o = shfl_up16(gv, d);
      if (int(lane) >= d) gv = stv16_compose(o, gv);
    }
    Stv16 gx = shfl_up16(gv, 1);
    if (lane == 0) gx = stv16_id();
    uint32_t g = stv16_apply(gx, gq);
    gq = __shfl_sync(FULL, stv16_apply(gv, gq), 31);
    // the segment's digits and signs, its states known
    uint32_t ni = 0, nf = 0, zl = 0xFFFFFFFFu, pzl = 0, szl = 0, pel = 0xFFFFFFFFu, sel = 0;
    bool mn = false, en = false;
    {
      uint32_t s = s_lane;
#pragma unroll
      for (uint32_t j = 0; j < LONG_SEG; ++j) {
        if (j >= len) continue;
        const uint32_t s_before = s;
        const uint32_t b = (bw[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        step_ctrl(lut, code_at(a + j, b), s);
        if (!((val_m >> j) & 1u)) continue;
        const uint32_t c = sym_class(b);
        const uint32_t ns = nib_apply(class_vec(c), g);
        if (c == 0) {
          if (ns == G2 || ns == G4) {
            if (b != '0' && zl == 0xFFFFFFFFu) { zl = ni + nf; pzl = j; szl = s_before; }
            if (ns == G2) ++ni; else ++nf;
          } else if (ns == G7 && b != '0' && pel == 0xFFFFFFFFu) {
            pel = j; sel = s_before;
          }
        } else if (c == 1 && b == '-') {
          if (ns == G1) mn = true;
          else if (ns == G6) en = true;
        }
        g = ns;
      }
    }
    // combine the lanes: digit indexes, first non-zero digits, counts
    uint32_t md = ni + nf;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, md, d);
      if (int(lane) >= d) md += o;
    }
    const uint32_t md_before = md - (ni + nf);
    if (z == NONE) {
      const uint64_t cand = zl != 0xFFFFFFFFu ? n_int + n_frac + md_before + zl : NONE;
      const uint64_t m = warp_min64(cand);
      if (m != NONE) {
        const uint32_t src = __ffs(__ballot_sync(FULL, cand == m)) - 1;
        z = m;
        pz = __shfl_sync(FULL, a + pzl, src);
        sz = __shfl_sync(FULL, szl, src);
      }
    }
    if (pez == NONE) {
      const uint64_t cand = pel != 0xFFFFFFFFu ? a + pel : NONE;
      const uint64_t m = warp_min64(cand);
      if (m != NONE) {
        const uint32_t src = __ffs(__ballot_sync(FULL, cand == m)) - 1;
        pez = m;
        sez = __shfl_sync(FULL, sel, src);
      }
    }
    n_int += __reduce_add_sync(FULL, ni);
    n_frac += __reduce_add_sync(FULL, nf);
    n_val += __reduce_add_sync(FULL, uint32_t(__popc(val_m)));
    mneg |= __any_sync(FULL, mn);
    eneg |= __any_sync(FULL, en);
  }
  if (lane != 0) return;
  uint64_t val = P.defval[col];
  int err = 0;
  if (n_val) {
    const bool accept = ty == PP_COL_FLOAT64 ? (gq == G2 || gq == G4 || gq == G7) : gq == G2;
    const uint64_t L = n_int + n_frac;
    val = 0;
    if (!accept) {
      err = PP_ERR_NUM_SYNTAX;
    } else if (ty != PP_COL_FLOAT64 && z != NONE && L - z > 19) {
      err = PP_ERR_NUM_OVERFLOW;  // 20 or more significant digits
    } else {
      // the significant digits, at most 19, from the first non-zero one
      uint64_t m = 0;
      if (z != NONE) {
        const uint64_t want = min(L - z, uint64_t(19));
        uint64_t got = 0;
        uint32_t s = sz;
        for (uint64_t p = pz; p < ge && got < want; ++p) {
          const uint32_t b = __ldg(P.in + p);
          if (step_ctrl(lut, code_at(p, b), s)) continue;
          if (b - '0' <= 9u) { m = m * 10 + (b - '0'); ++got; }
        }
      }
      if (ty == PP_COL_FLOAT64) {
        uint64_t mag = 0;
        if (z != NONE) {
          // the exponent: at most 7 significant digits, saturated above 100000
          int64_t ex = 0;
          if (pez != NONE) {
            uint32_t s = sez;
            for (uint64_t p = pez; p < ge && ex <= 100000; ++p) {
              const uint32_t b = __ldg(P.in + p);
              if (step_ctrl(lut, code_at(p, b), s)) continue;
              ex = ex * 10 + int64_t(b - '0');
            }
          }
          const uint64_t q = min(z + 19, L);
          const int64_t d10 = -int64_t(q > n_int ? q - n_int : 0) +
                              int64_t(n_int > z + 19 ? n_int - z - 19 : 0);
          int64_t e10 = d10 + (eneg ? -ex : ex);
          e10 = max(int64_t(-0x40000000), min(int64_t(0x40000000), e10));
          mag = ppn::decimal_to_binary64(m, int(e10));
        }
        val = mag | (mneg ? (1ull << 63) : 0ull);
      } else {
        const uint64_t lim = ty == PP_COL_INT8 ? 127ull : ty == PP_COL_INT32 ? 2147483647ull
                                                                             : 9223372036854775807ull;
        if (m > lim + (mneg ? 1u : 0u)) err = PP_ERR_NUM_OVERFLOW;
        else val = mneg ? ~m + 1 : m;
      }
    }
  }
  void* const out = P.typed[col];
  if (ty == PP_COL_INT32) static_cast<int32_t*>(out)[f.rec] = int32_t(val);
  else if (ty == PP_COL_INT8) static_cast<int8_t*>(out)[f.rec] = int8_t(val);
  else static_cast<uint64_t*>(out)[f.rec] = val;
  if (err) report(P.st, err, gs, true);
}

// Fields converted by long_field_kernel on this device (a test hook's count).
__device__ unsigned long long g_long_fields;

// The queued long fields, a warp each.
__global__ void __launch_bounds__(LF_NT) long_field_kernel(const __grid_constant__ ParseParams P) {
  __shared__ uint32_t lut[256];
  for (int k = threadIdx.x; k < 256; k += LF_NT) lut[k] = P.lut[k];
  __syncthreads();
  // the queue proper, then (with an encoding) the fields begun in an earlier tile
  const uint32_t n1 = min(P.s.counters[4], P.s.long_cap), n = n1 + P.s.counters[5];
  if (blockIdx.x == 0 && threadIdx.x == 0 && n) atomicAdd(&g_long_fields, n);
  const uint32_t warps = gridDim.x * (LF_NT / 32);
  for (uint32_t q = blockIdx.x * (LF_NT / 32) + (threadIdx.x >> 5); q < n; q += warps)
    convert_long(P, lut, P.s.long_q[q < n1 ? q : P.s.long_cap + (q - n1)]);
}

// ------------------------------------------------------ type inference
// The smallest type backing a field's value (ParPaRaw Section 4, "Type
// inference"): 1 int8, 2 int32, 3 int64, 4 float64 (also an integer beyond
// int64), 5 string; 0 for an empty or missing field.  Both number grammars
// read the value bytes at once.
struct TypeAcc {
  ppn::IntAcc i;
  ppn::FloatAcc f;
  __device__ __forceinline__ void feed(uint32_t c) { i.feed(c); f.feed(c); }
};
__device__ __forceinline__ uint32_t infer_field(const ParseParams& P, uint32_t v, const NumCtx& X) {
  if (v == SLOT_DEFAULT) return 0;
  const uint32_t fsr = v >> 16, fe = v & 0xFFFFu;
  TypeAcc acc;
  const uint32_t nd = feed_field(acc, P, fsr == 0xFFFFu ? X.tile_fstart : X.tile_base + fsr,
                                 X.tile_base + fe, X.tile_base, X.tile_s, X.ctrl_s, X.lut,
                                 X.tile_fstate);
  if (!nd) return 0;
  int64_t x;
  const int rc = acc.i.finish(128ull, 127ull, &x);
  if (rc == 0) return 1;
  if (rc == PP_ERR_NUM_OVERFLOW) {
    if (acc.i.finish(2147483648ull, 2147483647ull, &x) == 0) return 2;
    if (acc.i.finish(9223372036854775808ull, 9223372036854775807ull, &x) == 0) return 3;
    return 4;
  }
  uint64_t b;
  return acc.f.finish(&b) == 0 ? 4u : 5u;
}

__global__ void infer_finish_kernel(const uint32_t* codes, int32_t* types, int n) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n) return;
  static constexpr int32_t kind[6] = {PP_COL_INT8, PP_COL_INT8, PP_COL_INT32, PP_COL_INT64,
                                      PP_COL_FLOAT64, PP_COL_STRING};
  types[c] = kind[min(codes[c], 5u)];
}

// ------------------------------------------------ dropped records (pp_parse_ex)
__device__ __forceinline__ bool rec_dropped(const ParseParams& P, uint64_t rec) {
  return (P.drop_bits[rec >> 5] >> (rec & 31u)) & 1u;
}
// dropped records before record `rec`
__device__ __forceinline__ uint64_t dropped_before(const ParseParams& P, uint64_t rec) {
  const uint64_t g = rec >> 8, w = rec >> 5;
  uint64_t d = P.drop_pre[g];
  for (uint64_t k = g << 3; k < w; ++k) d += __popc(P.drop_bits[k]);
  const uint32_t b = uint32_t(rec & 31u);
  if (b) d += __popc(P.drop_bits[w] & ((1u << b) - 1u));
  return d;
}
// record `rec` is on the caller's skip list (skipped records are not checked)
__device__ __forceinline__ bool rec_skip_listed(const ParseParams& P, uint64_t rec) {
  uint64_t lo = 0, hi = P.n_skip;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) >> 1;
    if (P.skip_list[mid] < rec) lo = mid + 1;
    else hi = mid;
  }
  return lo < P.n_skip && P.skip_list[lo] == rec;
}

// ================================================================ 1. tile pass
// Everything after the tile start states happens in one pass over the tiles.
// A block has 16 worker warps (one 32-byte chunk per thread, as in the tile
// states pass), a context warp and, with string columns, a chars warp.  The
// two run the cross-tile exclusive scans of ParPaRaw Section 3.2 as
// single-pass decoupled look-backs, the context warp (record count, column
// offset, last terminator) and the chars warp the value bytes per string
// column, while the workers go on with the tile's own work; named barriers
// hand the aggregates and the prefixes between the roles:
//
//   workers                                   context / chars warp
//   tag the tile, scan it        --BAR_AGG-->  post the tile's aggregate,
//   list its fields (rows and                  look back: record index,
//   columns inside the tile),                  column and last terminator
//   value bytes per string                     at the tile start
//   column                       --BAR_W2--->
//   place the first record's     <--BAR_V2---  post the chars aggregate,
//   fields; stage strings,                     look back: chars offsets
//   convert numbers (stored at                 of the tile
//   their global rows)           <--BAR_CHR--
//   write offsets and chars
//
// A tile of one pass of rows (the plain kernel) writes its offsets and chars
// during the next tile instead, after that tile's field walk: its chars
// look-back has finished by then.  Such a tile also hands the chars warp its
// value bytes per string column only after the string items scan (the
// column totals of that scan), so its field walk counts none.

// The first record of a tile (its row 0) is in general the tail of a record
// that began earlier: its fields' columns are the tile's entry column plus
// their index, known only from the look-back (ParPaRaw Section 3.2, the
// "relative" column offset), so the workers keep them aside by index until
// then.  Tiles are handed out by an atomic ticket, so a tile's predecessors
// have always been started; a block takes its next ticket and starts that
// tile's copy late in the current tile (after the number conversions), so
// that tiles start in about ticket order and a tile's predecessors have
// mostly posted their aggregates by the time it looks back.
constexpr int BUF_BYTES = TILE + 64;      // landing buffer: the tile at toff, slack for word reads
constexpr uint32_t SHORT_FIELD = 32;      // longer string fields are staged chunk-parallel
constexpr uint16_t NO_FIELD = 0xFFFFu;
constexpr uint32_t REL_START = 0xFFFFu;   // slot start: the field began before the tile
constexpr uint32_t BAR_W = 1, BAR_AGG = 2, BAR_W2 = 3, BAR_V2 = 4, BAR_CHR = 5;
constexpr uint64_t M40 = (1ull << 40) - 1;
constexpr uint32_t COL_SAT = 0x1FFF00u;   // column counts saturate here (fit the look-back descriptor)

__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// The tile's bytes sit at buf[toff + p], toff = the input's address mod 16,
// so the 16-byte aligned span [c0, c1) of the tile (tile coordinates, c0 may
// be negative: bytes of the tile before) lands by one bulk copy at a 16-byte
// aligned buffer address.  The span never leaves the input; plain loads fill
// [0, c0) (the first tile of a misaligned input) and [c1, len) (the end of
// the input).  c1 <= c0: no bulk copy.
struct Span { int32_t c0, c1; };
__device__ __forceinline__ Span bulk_span(const ParseParams& P, uint32_t tile, uint32_t toff) {
  const uint64_t base = reinterpret_cast<uintptr_t>(P.in);
  const uint64_t tb = uint64_t(tile) * TILE;
  const uint32_t len = uint32_t(min(uint64_t(TILE), P.n - tb));
  const uint64_t a = base + tb, end = base + P.n;
  uint64_t lo = a - toff;
  if (lo < base) lo += 16;
  uint64_t hi = (a + len + 15) & ~uint64_t(15);
  if (hi > end) hi = (a + len) & ~uint64_t(15);
  if (hi <= lo) return {0, 0};
  return {int32_t(int64_t(lo) - int64_t(a)), int32_t(int64_t(hi) - int64_t(a))};
}

// Start the bulk copy of `tile` into buf (one elected thread); 1 if started.
__device__ __forceinline__ uint32_t issue_span(const ParseParams& P, uint32_t tile, uint32_t toff,
                                               uint8_t* buf, uint64_t* bar) {
  if (tile >= P.n_tiles) return 0;
  const Span s = bulk_span(P, tile, toff);
  if (s.c1 <= s.c0) return 0;
  const uint32_t bytes = uint32_t(s.c1 - s.c0);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(buf + int32_t(toff) + s.c0, P.in + int64_t(uint64_t(tile) * TILE) + s.c0, bytes, bar);
  return 1;
}

// This thread's 32 bytes of the tile.
__device__ __forceinline__ void load_chunk(const uint8_t* buf, uint32_t toff, uint32_t t,
                                           uint32_t (&w)[8]) {
  if (toff == 0) {
    const uint4* src = reinterpret_cast<const uint4*>(buf + t * CB);
    const int sw = (t >> 2) & 1;  // alternate read order: conflict-free 16-byte reads
    const uint4 x = src[sw], y = src[sw ^ 1];
    const uint4 lo = sw ? y : x, hi = sw ? x : y;
    w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
    w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
  } else {
    const uint32_t* rw = reinterpret_cast<const uint32_t*>(buf);
    const uint32_t a = t * CB + toff, q = a >> 2, sh = (a & 3u) * 8u;
    uint32_t r[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) r[k] = rw[q + k];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __funnelshift_r(r[k], r[k + 1], sh);
  }
}

// Chunk vectors composed over the worker warps (block_stv with the workers'
// barrier).
// wex: the composition of the warps before this one, which every warp
// computes itself after the one barrier.
__device__ __forceinline__ uint32_t block_stv_w(uint32_t G, uint32_t* warp_stv, uint32_t& wex) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = G;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, inc, d);
    if (lane >= d) inc = stv_compose(o, inc);
  }
  uint32_t lane_ex = __shfl_up_sync(FULL, inc, 1);
  if (lane == 0) lane_ex = STV_ID;
  if (lane == 31) warp_stv[warp] = inc;
  bar_sync(BAR_W, NT);
  uint32_t wi = lane < warp ? warp_stv[lane] : STV_ID;
#pragma unroll
  for (int d = 1; d < NW; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, wi, d);
    if (lane >= d) wi = stv_compose(o, wi);
  }
  wex = __shfl_sync(FULL, wi, warp > 0 ? warp - 1 : 0);
  if (warp == 0) wex = STV_ID;
  return lane_ex;
}

// (record count, last terminator as a global position + 1, column | state
// after the last terminator << 32): the record-count and column-offset
// operators of ParPaRaw Section 3.2, for the cross-tile look-back.
struct V2Op {
  __device__ void operator()(const uint64_t (&a)[3], const uint64_t (&b)[3],
                             uint64_t (&o)[3]) const {
    o[0] = a[0] + b[0];
    const bool hb = b[1] != 0;
    o[1] = hb ? b[1] : a[1];
    const uint32_t ac = uint32_t(a[2]), bc = uint32_t(b[2]);
    uint32_t col;
    if (bc & ABS32) {
      col = bc;
    } else {
      const uint64_t s = uint64_t(ac & ~ABS32) + bc;
      col = (ac & ABS32) | uint32_t(s > COL_SAT ? uint64_t(COL_SAT) : s);
    }
    o[2] = uint64_t(col) | (uint64_t(hb ? uint32_t(b[2] >> 32) : uint32_t(a[2] >> 32)) << 32);
  }
};

// The context look-back's per-tile descriptor: two 64-bit words, each
// carrying the status in bits 0..1 (none / aggregate / inclusive prefix),
// so that one 16-byte load reads a whole descriptor and a descriptor whose
// two words show different statuses (read while being rewritten) counts as
// not posted yet.
//   word 0: status | records << 2 (40 bits) | state after the last terminator << 42
//   word 1: status | (last terminator + 1) << 2 (40 bits) | column << 42
// The column takes 22 bits: bit 21 absolute, 21 bits of count, saturated
// (a record's fields beyond n_cols <= 64 are dropped anyway).  Positions and
// record counts stay below 2^40 (inputs are limited to 2^40 bytes).
__device__ __forceinline__ uint32_t col_pack(uint32_t c) {
  return ((c & ABS32) ? (1u << 21) : 0u) | min(c & ~ABS32, COL_SAT);
}
__device__ __forceinline__ uint32_t col_unpack(uint32_t c) {
  return ((c >> 21) & 1u ? ABS32 : 0u) | (c & 0x1FFFFFu);
}
__device__ __forceinline__ void v2_pack(uint32_t flag, const uint64_t (&v)[3], uint64_t& w0,
                                        uint64_t& w1) {
  w0 = flag | ((v[0] & M40) << 2) | (uint64_t(uint32_t(v[2] >> 32) & 0xFu) << 42);
  w1 = flag | ((v[1] & M40) << 2) | (uint64_t(col_pack(uint32_t(v[2]))) << 42);
}
__device__ __forceinline__ void v2_unpack(uint64_t w0, uint64_t w1, uint64_t (&v)[3]) {
  v[0] = (w0 >> 2) & M40;
  v[1] = (w1 >> 2) & M40;
  v[2] = uint64_t(col_unpack(uint32_t(w1 >> 42))) | (uint64_t((w0 >> 42) & 0xFu) << 32);
}
__device__ __forceinline__ void st_v2desc(uint64_t* d, uint64_t w0, uint64_t w1) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(d), "l"(w0), "l"(w1) : "memory");
}
__device__ __forceinline__ void ld_v2desc(const uint64_t* d, uint64_t& w0, uint64_t& w1) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(d) : "memory");
}

// Decoupled look-back over the descriptors (one full warp): posts the
// tile's aggregate, returns its exclusive prefix and posts its inclusive
// prefix.  Every wait is bounded; a wait that runs out reports
// PP_ERR_LOOKBACK_TIMEOUT and takes the missing tiles as empty.
__device__ void v2_lookback(uint64_t* desc, uint32_t tile, const uint64_t (&agg)[3],
                            const LookbackCfg& cfg, uint64_t (&out_excl)[3]) {
  const int lane = threadIdx.x & 31;
  const V2Op op;
  const uint64_t seed[3] = {0ull, 0ull, uint64_t(ABS32)};
  const uint64_t ident[3] = {0ull, 0ull, 0ull};
  uint64_t w0, w1;
  if (tile == 0) {
    uint64_t inc[3];
    op(seed, agg, inc);
    v2_pack(LB_INC, inc, w0, w1);
    if (lane == 0) st_v2desc(desc, w0, w1);
#pragma unroll
    for (int k = 0; k < 3; ++k) out_excl[k] = seed[k];
    return;
  }
  v2_pack(LB_AGG, agg, w0, w1);
  if (lane == 0) st_v2desc(desc + 2 * size_t(tile), w0, w1);
  uint64_t acc[3] = {0ull, 0ull, 0ull};
  int64_t base = int64_t(tile) - 1;
  uint32_t spins = 0;
  bool timed_out = false;
  for (;;) {
    const int64_t idx = base - lane;
    uint32_t f;
    uint64_t v[3];
    for (;;) {
      if (idx >= 0) {
        ld_v2desc(desc + 2 * size_t(idx), w0, w1);
        f = uint32_t(w0 & 3u) == uint32_t(w1 & 3u) ? uint32_t(w0 & 3u) : LB_NONE;
      } else {
        f = LB_INC;
      }
      if (lb_ready(f)) break;
      if (!lb_backoff(spins, cfg.spin_limit)) { timed_out = true; break; }
    }
    if (idx < 0) {
#pragma unroll
      for (int k = 0; k < 3; ++k) v[k] = seed[k];
    } else if (f == LB_NONE) {  // only after a timeout
#pragma unroll
      for (int k = 0; k < 3; ++k) v[k] = ident[k];
      f = LB_INC;
    } else {
      v2_unpack(w0, w1, v);
    }
    const uint32_t pmask = __ballot_sync(FULL, f == LB_INC);
    const int stop = pmask ? __ffs(pmask) - 1 : 31;
    if (lane > stop) {
#pragma unroll
      for (int k = 0; k < 3; ++k) v[k] = ident[k];
    }
    // lane L combines with lane L+d, which holds an EARLIER tile
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint64_t o[3], t[3];
#pragma unroll
      for (int k = 0; k < 3; ++k) o[k] = __shfl_down_sync(FULL, v[k], d);
      if (lane + d < 32) {
        op(o, v, t);
#pragma unroll
        for (int k = 0; k < 3; ++k) v[k] = t[k];
      }
    }
    uint64_t r[3], t[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) r[k] = __shfl_sync(FULL, v[k], 0);
    op(r, acc, t);
#pragma unroll
    for (int k = 0; k < 3; ++k) acc[k] = t[k];
    if (pmask) break;
    base -= 32;
  }
  if (timed_out && lane == 0) report(cfg.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
  uint64_t inc[3];
  op(acc, agg, inc);
  v2_pack(LB_INC, inc, w0, w1);
  if (lane == 0) st_v2desc(desc + 2 * size_t(tile), w0, w1);
#pragma unroll
  for (int k = 0; k < 3; ++k) out_excl[k] = acc[k];
}

struct PShared {
  uint64_t bar[2];               // landing buffers' mbarriers
  uint32_t tile[2];              // ticket per buffer (written by the scan warp)
  uint32_t issued[2], wpar[2];   // bulk copy started, phase parity to wait for
  uint32_t warp_stv[NW];
  uint32_t wv[NW][3];            // per warp (records, column, last), then exclusive
  uint32_t wc[NW + 1];           // control bytes per warp, then exclusive; [NW] = tile total
  uint32_t wrd[NW];              // partial mode: 1 + the warp's last record delimiter
  uint32_t agg_rec, agg_col, agg_last, n_ctrl, virt;  // the tile's totals
  uint32_t rel_slot[PP_MAX_COLS];  // row-0 field k: slot value
  uint32_t rel_len[PP_MAX_COLS];   // row-0 field k: value bytes
  uint32_t n_rel;                  // row-0 fields seen (k + 1 of the last)
  uint32_t rd0_pos, rd0_k;         // the tile's first record delimiter: position + 1, field index
  uint32_t ctot[ppi::MAX_STR_COLS];  // value bytes per string column of rows >= 1
  uint32_t cmode[2];               // per landing buffer: 1 = the chars aggregate is the
                                   // items scan's column totals (a one-pass tile)
  uint64_t rec0, last1;            // from the look-back: record index, last terminator + 1
  uint32_t col_in, lst;            // column at the tile start, state after that terminator
  uint64_t base[ppi::MAX_STR_COLS];  // chars offset of the tile per string column
  uint32_t wsum[NW];
  uint32_t cstart[ppi::MAX_STR_COLS + 1];  // staging start per string column (this pass)
  uint32_t carry[ppi::MAX_STR_COLS];       // chars of earlier passes per string column
  uint32_t wo_len[ppi::MAX_STR_COLS], wo_head[ppi::MAX_STR_COLS];  // chars write-out per column:
  uint32_t wo_vpre[ppi::MAX_STR_COLS + 1];  // bytes, head bytes, 16-byte middles before it
  uint64_t pd_rec0;                // deferred write-out: the tile's first record,
  uint32_t pd_rows, pd_col_in, pd_col_end;  // its rows, entry and end columns
  uint8_t coltype[PP_MAX_COLS];
  uint8_t numcol[PP_MAX_COLS];     // numeric output columns, floats first
  uint32_t n_num;
  uint32_t lut1[256];              // the LUT, one entry per byte value
  uint8_t sym_b2g[0x80];           // encodings: groups of the code points below 0x80
  uint32_t inf[PP_MAX_COLS];       // type inference: largest type code per column
  uint16_t cpl[NT + 1];            // control bytes before chunk t inside its warp
  uint16_t lk[2][NT];              // long string field (item) continuing in / starting in chunk t
};
constexpr size_t PARSE_SMEM = LUT_BYTES + 2 * BUF_BYTES + STAGE_BYTES + SLOT_CAP * 4 + NT * 4 +
                              SLOT_CAP * 2 + sizeof(PShared);

// control bytes of the tile before position p (p <= tile length)
__device__ __forceinline__ uint32_t ctrl_bef(const uint32_t* ctrl_s, const PShared& S, uint32_t p) {
  const uint32_t c = p >> 5, b = p & 31u;
  return S.wc[c >> 5] + S.cpl[c] + (b ? uint32_t(__popc(ctrl_s[c] & ((1u << b) - 1u))) : 0u);
}
// Copy tile bytes [p, p + len) to dst[d ...] (staging): bytes up to the
// next 4-byte boundary of the destination, then whole words built from two
// source words by a funnel shift (raw_w: the landing buffer as words, tile
// byte p at byte p + toff; it has slack for the word after the last), then
// the last bytes.
__device__ __forceinline__ void copy_run(uint8_t* dst, uint32_t d, const uint8_t* tile_s,
                                         const uint32_t* raw_w, uint32_t toff, uint32_t p,
                                         uint32_t len) {
  for (; len && (d & 3u); --len) dst[d++] = tile_s[p++];
  const uint32_t nw = len >> 2;
  if (nw) {
    uint32_t* dw = reinterpret_cast<uint32_t*>(dst + d);
    const uint32_t a = p + toff, sh = (a & 3u) * 8u;
    const uint32_t* sw = raw_w + (a >> 2);
    uint32_t lo = sw[0];
    for (uint32_t i = 0; i < nw; ++i) {
      const uint32_t hi = sw[i + 1];
      dw[i] = __funnelshift_r(lo, hi, sh);
      lo = hi;
    }
    d += 4 * nw;
    p += 4 * nw;
    len -= 4 * nw;
  }
  for (; len; --len) dst[d++] = tile_s[p++];
}

// value bytes of the field [fs, e) inside the tile (fs = REL_START: from 0)
__device__ __forceinline__ uint32_t value_len(uint32_t fs, uint32_t e, bool any_ctrl,
                                              const uint32_t* ctrl_s, const PShared& S) {
  const uint32_t a0 = fs == REL_START ? 0u : fs;
  return (e - a0) - (any_ctrl ? ctrl_bef(ctrl_s, S, e) - ctrl_bef(ctrl_s, S, a0) : 0u);
}

// ------------------------------------------------------------- scan warps
// Block sizes: the workers, the context warp, and (with string columns) the
// chars warp.
template <int NS>
__host__ __device__ constexpr int ntf_of() { return NT + (NS > 0 ? 64 : 32); }

// The context warp: per tile, the record/column look-back.
template <int NS>
__device__ void ctx_role(const ParseParams& P, PShared& S) {
  constexpr uint32_t NTF_ = ntf_of<NS>();
  const int lane = threadIdx.x & 31;
  const LookbackCfg cfg{P.st, P.spin_limit};
  for (uint32_t it = 0;; ++it) {
    const uint32_t b = it & 1u;
    bar_sync(BAR_AGG, NT + 32);  // the workers' tile aggregate (or their exit)
    const uint32_t tile = S.tile[b];
    if (tile >= P.n_tiles) {
      bar_arrive(BAR_V2, NTF_);  // the last barrier the other roles wait on
      break;
    }
    const uint64_t tile_base = uint64_t(tile) * TILE;
    uint64_t agg[3], ex[3];
    agg[0] = S.agg_rec;
    agg[1] = S.agg_last ? tile_base + (S.agg_last >> 8) : 0ull;
    agg[2] = uint64_t(S.agg_col) | (uint64_t(S.agg_last & 0xFFu) << 32);
    if (P.dbg_withhold && tile == 0) {  // test hook: post nothing, later tiles time out
      ex[0] = 0; ex[1] = 0; ex[2] = ABS32;
    } else {
      v2_lookback(P.s.v2_desc, tile, agg, cfg, ex);
    }
    if (lane == 0) {
      S.rec0 = ex[0];
      S.last1 = ex[1];
      S.col_in = uint32_t(ex[2]) & ~ABS32;
      S.lst = uint32_t(ex[2] >> 32);
    }
    __syncwarp();
    bar_arrive(BAR_V2, NTF_);
  }
}

// The chars warp: per tile, the chars aggregate (its first record's fields
// placed by the entry column) and the chars look-back.
template <int NS>
__device__ void chars_role(const ParseParams& P, PShared& S) {
  constexpr int K3 = NS > 0 ? NS : 1;
  constexpr uint32_t NTF_ = ntf_of<NS>();
  const int lane = threadIdx.x & 31;
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t n_cols = uint32_t(P.n_cols);
  for (uint32_t it = 0;; ++it) {
    const uint32_t b = it & 1u;
    bar_sync(BAR_V2, NTF_);     // the entry column (or the workers' exit)
    const uint32_t tile = S.tile[b];
    if (tile >= P.n_tiles) break;
    bar_sync(BAR_W2, NT + 32);  // the workers' value-byte totals
    uint64_t cagg[K3];
    if (S.cmode[b]) {  // a one-pass tile: the column totals of its items scan
#pragma unroll
      for (int k = 0; k < K3; ++k) cagg[k] = k < P.n_str ? uint64_t(S.cstart[k + 1] - S.cstart[k]) : 0u;
    } else {  // the field walk's totals of rows >= 1, and row 0's fields
      const uint32_t col_in = S.col_in;
      const uint32_t nrel = min(S.n_rel, n_cols);
#pragma unroll
      for (int k = 0; k < K3; ++k) cagg[k] = k < P.n_str ? S.ctot[k] : 0u;
      // row-0 fields: column = entry column + index (at most n_cols of them,
      // summed by one lane and broadcast)
      uint32_t add[K3];
#pragma unroll
      for (int q = 0; q < K3; ++q) add[q] = 0;
      if (lane == 0)
        for (uint32_t k = 0; k < nrel && col_in + k < n_cols; ++k) {
          const int si = P.stridx[col_in + k];
          const uint32_t len = S.rel_len[k];
#pragma unroll
          for (int q = 0; q < K3; ++q)
            if (q == si) add[q] += len;
        }
#pragma unroll
      for (int q = 0; q < K3; ++q) cagg[q] += __shfl_sync(FULL, add[q], 0);
    }
    uint64_t zero[K3], ex[K3];
#pragma unroll
    for (int k = 0; k < K3; ++k) zero[k] = 0;
    if (P.dbg_withhold && tile == 0) {
#pragma unroll
      for (int k = 0; k < K3; ++k) ex[k] = 0;
    } else {
      lookback_vec<K3>(P.s.c_flag, P.s.c_agg, P.s.c_inc, tile, cagg, zero, zero, AddOp<K3>{},
                       cfg, ex);
    }
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < K3; ++k)
        if (k < P.n_str) S.base[k] = ex[k];
      if (tile + 1 == P.n_tiles)  // the input's chars per string column
#pragma unroll
        for (int k = 0; k < K3; ++k)
          if (k < P.n_str) P.st->chars_len[P.strcol[k]] = ex[k] + cagg[k];
    }
    __syncwarp();
    bar_arrive(BAR_CHR, NT + 32);
  }
}

// ----------------------------------------------------------------- kernel
// GEN: the general kernel, for inputs in an encoding (symbol codes; see
// sym_code), the options of pp_parse_ex, type inference, streamed chunks
// (partial mode) and the tag test hook; the plain kernel (a whole byte
// input, every record emitted) carries none of that code.
template <int NS, bool GEN>
__global__ void __launch_bounds__(ntf_of<NS>(), 2) parse_kernel(const __grid_constant__ ParseParams P) {
  constexpr int NTF = ntf_of<NS>();
  constexpr int NSW = NS > 0 ? (NS + 3) / 4 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin0 = smem + LUT_BYTES;  // two landing buffers
  uint8_t* stage_s = lin0 + 2 * BUF_BYTES;
  uint32_t* slot_s = reinterpret_cast<uint32_t*>(stage_s + STAGE_BYTES);
  uint32_t* ctrl_s = slot_s + SLOT_CAP;
  uint16_t* pos_s = reinterpret_cast<uint16_t*>(ctrl_s + NT);  // chars end per string field
  PShared& S = *reinterpret_cast<PShared*>(pos_s + SLOT_CAP);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t toff = uint32_t(reinterpret_cast<uintptr_t>(P.in) & 15u);
  for (int k = t; k < 256 * 32; k += NTF) lut_s[k] = P.lut[k >> 5];
  for (int k = t; k < 256; k += NTF) S.lut1[k] = P.lut[k];
  for (int k = t; k < 0x80; k += NTF) S.sym_b2g[k] = P.sym_b2g[k];
  if (t < PP_MAX_COLS) { S.coltype[t] = P.coltype[t]; S.inf[t] = 0; }
  if (t < ppi::MAX_STR_COLS) S.carry[t] = 0;
  if (t == 0) {
    uint32_t m = 0;
    for (uint32_t c = 0; c < uint32_t(P.n_cols); ++c)
      if (P.coltype[c] == PP_COL_FLOAT64) S.numcol[m++] = uint8_t(c);
    for (uint32_t c = 0; c < uint32_t(P.n_cols); ++c)  // the integer columns after the floats
      if (P.coltype[c] != PP_COL_SKIP && P.coltype[c] != PP_COL_STRING &&
          P.coltype[c] != PP_COL_FLOAT64)
        S.numcol[m++] = uint8_t(c);
    S.n_num = P.has_out ? m : 0u;
    S.cpl[NT] = 0;
  }
  if (warp == NW && lane == 0) {  // the first ticket and its copy
    mbar_init(&S.bar[0], 1);
    mbar_init(&S.bar[1], 1);
    const uint32_t first = atomicAdd(&P.s.counters[0], 1u);
    S.tile[0] = first;
    S.issued[0] = issue_span(P, first, toff, lin0, &S.bar[0]);
    S.wpar[0] = 0;
    S.tile[1] = 0xFFFFFFFFu;
    S.issued[1] = 0;
    S.wpar[1] = 0;
  }
  __syncthreads();
  if (warp == NW) {
    ctx_role<NS>(P, S);
    return;
  }
  if (warp == NW + 1) {
    chars_role<NS>(P, S);
    return;
  }

  const uint32_t* my_lut = lut_s + lane;
  const uint32_t n_cols = uint32_t(P.n_cols);
  const uint32_t n_str = NS > 0 ? uint32_t(P.n_str) : 0u;
  const uint32_t rpb = max(1u, (uint32_t(SLOT_CAP) - n_cols) / n_cols);  // rows per pass
  const bool partial = GEN && P.record_end != nullptr;  // a streamed chunk
  const bool emit = GEN && P.drop_bits != nullptr;    // some records are not emitted
  const bool status = GEN && P.mark_bits != nullptr;  // the status pass of rejection
  const bool infer = GEN && P.infer_out != nullptr;   // type inference
  // status pass: rows of the tile with a wrong field count (pos_s's space,
  // which only string staging uses)
  uint32_t* const flags_s = reinterpret_cast<uint32_t*>(pos_s);

  uint32_t nph[2] = {S.issued[0], 0u};  // thread 0: bulk copies started per buffer
  // The next tile's ticket and bulk copy (thread 0), taken late in the
  // current tile so that tiles start in ticket order and a tile's
  // predecessors have posted their aggregates when it looks back; the copy
  // goes to the buffer of the tile before, which is no longer read.
  auto next_ticket = [&](uint32_t b) {
    if (t != 0) return;
    const uint32_t o = b ^ 1u;
    const uint32_t nt = atomicAdd(&P.s.counters[0], 1u);
    const uint32_t iss = issue_span(P, nt, toff, lin0 + o * BUF_BYTES, &S.bar[o]);
    S.tile[o] = nt;
    S.issued[o] = iss;
    S.wpar[o] = nph[o] & 1u;
    nph[o] += iss;
  };

  // Arrow offsets and chars of the string fields of rows [lo, hi) of a tile
  // with `rows` rows, first record rec0, entry column col_in and end column
  // col_end, from the chars positions (pos_s), the column starts (S.cstart)
  // and the staged bytes; the column's chars begin at S.base + S.carry.
  auto write_out = [&](uint32_t lo, uint32_t hi, uint32_t rows, uint64_t rec0, uint32_t col_in,
                       uint32_t col_end) {
    const uint32_t nr = hi - lo, ngr = (nr + 31) / 32;
    const uint32_t n_str = NS > 0 ? uint32_t(P.n_str) : 0u;
    // Arrow offsets of the string fields closed in this pass
    uint32_t si = 0, gi = uint32_t(warp);
    while (gi >= ngr && si < n_str) { gi -= ngr; ++si; }
    for (; si < n_str; gi += NW) {
      while (gi >= ngr && si < n_str) { gi -= ngr; ++si; }
      if (si >= n_str) break;
      const uint32_t r = lo + gi * 32 + lane;
      const uint32_t c = P.strcol[si];
      if (r >= hi || (r == 0 && c < col_in) || (r + 1 == rows && c >= col_end)) continue;
      uint64_t rec = rec0 + r;
      if (emit) {
        if (rec_dropped(P, rec)) continue;
        rec -= dropped_before(P, rec);
      }
      if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
      const uint64_t off = S.base[si] + S.carry[si] + (pos_s[si * nr + (r - lo)] - S.cstart[si]);
      if (off > 0x7FFFFFFFull || off > P.chars_cap[si]) report(P.st, PP_ERR_CAPACITY, 0, false);
      else P.offsets[si][rec + 1] = int32_t(off);
    }
    // staged chars -> HBM, the string columns together: each column's
    // bytes up to a 16-byte boundary of its destination (head) and after its
    // last whole 16 bytes (tail) by a warp per column, and the 16-byte
    // middles of all columns as one index space (wo_vpre: middles before
    // each column), realigned by funnel shifts
    static_assert(ppi::MAX_STR_COLS <= NW, "a warp per string column");
    if (warp == 0) {
      uint32_t nv = 0;
      if (uint32_t(lane) < n_str) {
        const uint32_t si = uint32_t(lane);
        uint32_t len = S.cstart[si + 1] - S.cstart[si];
        const uint64_t gb = S.base[si] + S.carry[si];
        if (len && gb + len > P.chars_cap[si]) {
          report(P.st, PP_ERR_CAPACITY, 0, false);
          len = gb >= P.chars_cap[si] ? 0u : uint32_t(P.chars_cap[si] - gb);
        }
        const uint32_t head =
            min(len, uint32_t((16u - (reinterpret_cast<uintptr_t>(P.chars[si] + gb) & 15u)) & 15u));
        S.wo_len[si] = len;
        S.wo_head[si] = head;
        nv = (len - head) >> 4;
      }
      uint32_t inc = nv;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += o;
      }
      if (uint32_t(lane) < n_str) S.wo_vpre[lane + 1] = inc;
      if (lane == 0) S.wo_vpre[0] = 0;
    }
    bar_sync(BAR_W, NT);
    if (uint32_t(warp) < n_str) {
      const uint32_t si = uint32_t(warp), len = S.wo_len[si], head = S.wo_head[si];
      const uint32_t tail0 = head + (((len - head) >> 4) << 4), sp = S.cstart[si];
      uint8_t* gp = P.chars[si] + (S.base[si] + S.carry[si]);
      const uint32_t k = uint32_t(lane) & 15u;
      const uint32_t p = lane < 16 ? (k < head ? k : len) : tail0 + k;
      if (p < len) gp[p] = stage_s[sp + p];
    }
    const uint32_t vtot = S.wo_vpre[n_str];
    uint32_t vc = 0;  // the column of middle v
    for (uint32_t v = uint32_t(t); v < vtot; v += NT) {
      while (v >= S.wo_vpre[vc + 1]) ++vc;
      const uint32_t vi = v - S.wo_vpre[vc], head = S.wo_head[vc];
      const uint32_t src0 = S.cstart[vc] + head, sh = (src0 & 3u) * 8u;
      const uint32_t* q = reinterpret_cast<const uint32_t*>(stage_s + (src0 & ~3u)) + 4 * vi;
      const uint32_t a0 = q[0], a1 = q[1], a2 = q[2], a3 = q[3], a4 = q[4];
      uint4 o;
      o.x = __funnelshift_r(a0, a1, sh);
      o.y = __funnelshift_r(a1, a2, sh);
      o.z = __funnelshift_r(a2, a3, sh);
      o.w = __funnelshift_r(a3, a4, sh);
      __stcs(reinterpret_cast<uint4*>(P.chars[vc] + (S.base[vc] + S.carry[vc]) + head) + vi, o);
    }
  };
  // A tile of one pass in the plain kernel leaves its write-out pending
  // (pend) until the next tile has walked its fields: by then the chars
  // warp's look-back for it has long finished, where an immediate write-out
  // would wait for it.  The bytes stay staged meanwhile: the next tile
  // overwrites the staging area, the chars positions and the column starts
  // only after that.
  bool pend = false;

  for (uint32_t it = 0;; ++it) {
    const uint32_t b = it & 1u;
    const uint32_t tile = S.tile[b];
    if (tile >= P.n_tiles) {
      if (NS > 0 && pend) {  // the last tile's write-out
        bar_sync(BAR_CHR, NT + 32);
        write_out(0u, S.pd_rows, S.pd_rows, S.pd_rec0, S.pd_col_in, S.pd_col_end);
      }
      bar_arrive(BAR_AGG, NT + 32);  // the scan warps see the end too
      bar_sync(BAR_V2, NTF);
      break;
    }
    uint8_t* buf = lin0 + b * BUF_BYTES;
    const uint8_t* tile_s = buf + toff;
    const uint32_t* raw_w = reinterpret_cast<const uint32_t*>(buf);
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    const bool last_tile = tile + 1 == P.n_tiles;
    const uint32_t s_tile = P.s.tile_state[tile];
    if (t < ppi::MAX_STR_COLS) S.ctot[t] = 0;
    if (t < PP_MAX_COLS) S.rel_len[t] = 0;
    if (status)
      for (int q = t; q < (TILE + 32) / 32 + 1; q += NT) flags_s[q] = 0;
    if (t == 0) { S.n_rel = 0; S.rd0_pos = 0; S.rd0_k = 0; S.virt = 0; }

    // ---- the tile's bytes: bulk copy, plus plain loads at the input's ends
    {
      const uint32_t iss = S.issued[b];
      const Span sp = iss ? bulk_span(P, tile, toff) : Span{0, 0};
      if (iss && !mbar_wait_bounded(&S.bar[b], S.wpar[b], WAIT_LIMIT)) {
        if (t == 0) report(P.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
        mbar_wait_bounded(&S.bar[b], S.wpar[b], WAIT_LIMIT);
      }
      const uint32_t h0 = iss ? uint32_t(max(sp.c0, 0)) : tile_len;  // [0, h0) plain
      const uint32_t h1 = iss ? uint32_t(min(sp.c1, int32_t(tile_len))) : tile_len;
      if (h0 > 0 || h1 < tile_len) {
        for (uint32_t k = t; k < h0; k += NT) buf[toff + k] = P.in[tile_base + k];
        for (uint32_t k = h1 + t; k < tile_len; k += NT) buf[toff + k] = P.in[tile_base + k];
        bar_sync(BAR_W, NT);
      }
    }
    uint32_t w[8];
    load_chunk(buf, toff, uint32_t(t), w);
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    const uint8_t* own = tile_s + cstart;
    const uint8_t* dfa_s = tile_s;  // what the DFA reads: the bytes, or their symbol codes
    if (GEN && P.enc) {
      // a chunk of one-byte UTF-8 symbols is its own codes
      bool plain = P.enc == PP_ENC_UTF8 && clen == CB;
      if (plain) {
#pragma unroll
        for (int k = 0; k < 8; ++k) plain &= (w[k] & 0x80808080u) == 0;
        const uint64_t nx = tile_base + cstart + CB;
        if (plain && nx < P.n)
          plain = !is_cont(cstart + CB < tile_len ? uint32_t(tile_s[cstart + CB]) : uint32_t(__ldg(P.in + nx)));
      }
      if (!plain) {
        uint8_t* codes_s = stage_s;  // free until the strings are staged
        chunk_codes(P, S.sym_b2g, tile_s, tile_base, tile_len, cstart, clen, codes_s);
        if (clen == CB) {
          const uint4* c4 = reinterpret_cast<const uint4*>(codes_s + cstart);
          const uint4 x = c4[0], y = c4[1];
          w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
          w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
        }
        own = codes_s + cstart;
        dfa_s = codes_s;
      }
    }

    // ---- chunk start states and tags (ParPaRaw Section 3.1)
    uint32_t G, special, special_x;
    stv_pass(w, clen, dfa_s, cstart, my_lut, G, special, special_x);
    uint32_t warp_ex;
    const uint32_t lane_ex = block_stv_w(G, S.warp_stv, warp_ex);
    const uint32_t st = stv_apply(lane_ex, stv_apply(warp_ex, s_tile));
    const Tags g = tag_chunk(st, special, special_x, P.sticky, clen, cstart, own, my_lut,
                             P.bg_next);
    if (g.inv_at < clen && st != 4)
      report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + g.inv_at, true);
    const bool owns_end = last_tile && clen > 0 && cstart + clen == tile_len;
    const bool accepting = g.end != 4 && ((P.accept_mask >> g.end) & 1u);
    if (!partial && owns_end && g.end != 4 && !accepting)  // an invalid end is reported where it began
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    const bool virt_rd = !partial && owns_end && accepting && !((g.rd >> (clen - 1)) & 1u);
    const uint32_t fd = g.fd, rd = g.rd;
    ctrl_s[t] = g.ctrl;
    if (GEN && P.dbg_tags && clen) {  // test hook: the chunk's bitmaps
      uint32_t* o = P.dbg_tags + 3 * ((tile_base + cstart) / CB);
      o[0] = fd;
      o[1] = rd;
      o[2] = g.ctrl;
    }

    // ---- (records, column, last) and control bytes, scanned over the warp
    // and then over the warps
    V2 vi = chunk_v2(g);
    const uint32_t c_own = __popc(g.ctrl);
    uint32_t ci = c_own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const V2 o = shfl_up_v2(vi, d);
      const uint32_t oc = __shfl_up_sync(FULL, ci, d);
      if (lane >= d) {
        vi = op2_32(o, vi);
        ci += oc;
      }
    }
    V2 vex = shfl_up_v2(vi, 1);
    if (lane == 0) vex = {0u, 0u, 0u};
    if (lane == 31) {
      S.wv[warp][0] = vi.rec; S.wv[warp][1] = vi.col; S.wv[warp][2] = vi.last;
      S.wc[warp] = ci;
    }
    S.cpl[t] = uint16_t(ci - c_own);
    if (partial) {
      const uint32_t wm = __reduce_max_sync(FULL, rd ? cstart + 32u - __clz(rd) : 0u);
      if (lane == 0) S.wrd[warp] = wm;
    }
    if (virt_rd) S.virt = 1;
    bar_sync(BAR_W, NT);
    if (warp == 0) {
      V2 x = lane < NW ? V2{S.wv[lane][0], S.wv[lane][1], S.wv[lane][2]} : V2{0u, 0u, 0u};
      const uint32_t c0 = lane < NW ? S.wc[lane] : 0u;
      uint32_t xc = c0;
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const V2 o = shfl_up_v2(x, d);
        const uint32_t oc = __shfl_up_sync(FULL, xc, d);
        if (lane >= d) {
          x = op2_32(o, x);
          xc += oc;
        }
      }
      V2 xe = shfl_up_v2(x, 1);
      if (lane == 0) xe = {0u, 0u, 0u};
      __syncwarp();
      if (lane < NW) {
        S.wv[lane][0] = xe.rec; S.wv[lane][1] = xe.col; S.wv[lane][2] = xe.last;
        S.wc[lane] = xc - c0;
      }
      if (lane == NW - 1) {
        S.agg_rec = x.rec;
        S.agg_col = x.col;
        S.agg_last = x.last;
        S.n_ctrl = xc;
        S.wc[NW] = xc;
      }
      if (partial && lane == 0) {  // 1 + the tile's last record delimiter
        uint32_t m = 0;
        for (int q = 0; q < NW; ++q) m = max(m, S.wrd[q]);
        if (m) atomicMax(P.record_end, static_cast<unsigned long long>(tile_base + m));
      }
    }
    bar_sync(BAR_W, NT);
    bar_arrive(BAR_AGG, NT + 32);  // the context warp may post the tile's aggregate

    const V2 pre = op2_32(V2{S.wv[warp][0], S.wv[warp][1], S.wv[warp][2]}, vex);
    const bool any_ctrl = S.n_ctrl != 0;
    const bool any_virt = S.virt != 0;
    const uint32_t rows = S.agg_rec + 1;   // records touched by the tile (row 0: the one open at its start)
    const uint32_t rl0 = pre.rec;          // row at the chunk start
    const uint32_t col0 = pre.col & ~ABS32;  // column there; for row 0, the index in the row
    const uint32_t fs0 = pre.last ? (pre.last >> 8) : REL_START;  // start of the field open there
    const uint32_t term_all = fd | rd;
    const bool owns_tail = clen > 0 && cstart + clen == tile_len;

    // filled after the look-back
    uint64_t rec0 = 0;
    uint32_t col_in = 0, col_end = 0;
    // the conversion context; the field open at the tile start is known
    // only after the look-back, and only row 0 needs it
    NumCtx X{tile_base, 0ull, uint32_t(P.start_state), tile_s, raw_w, toff, ctrl_s, &S.wc[0],
             &S.cpl[0], &S.lut1[0], any_ctrl};


    // One pass of rows in the plain kernel: the write-out waits for the next
    // tile, and the chars aggregate is the items scan's column totals (the
    // field walk counts no value bytes)
    const bool defer = !GEN && P.has_out && rows <= rpb;
    if (t == 0) S.cmode[b] = defer ? 1u : 0u;
    // ---- fields -> (column, row) slots, in passes of rows
    for (uint32_t lo = 0; lo < rows; lo += rpb) {
      const uint32_t hi = min(rows, lo + rpb), nr = hi - lo;
      const uint32_t nrp = nr | 1u;  // odd stride: a warp's column-wise writes hit distinct banks
      const bool first = lo == 0;
      uint64_t cnt[NSW];  // value bytes per string column of rows >= 1 (packed 16-bit)
#pragma unroll
      for (int k = 0; k < NSW; ++k) cnt[k] = 0;
      if (NS > 0) { S.lk[0][t] = NO_FIELD; S.lk[1][t] = NO_FIELD; }
      // One field: row rl, column (row 0: index) col, tile span [fs, e).
      auto enter = [&](uint32_t rl, uint32_t col, uint32_t fs, uint32_t e, bool isrd, bool open) {
        const bool in_pass = rl - lo < nr;
        if (rl == 0) {
          if (first) {
            if (col < n_cols) {
              S.rel_slot[col] = (fs << 16) | e;
              if (!emit && !defer) {
                const uint32_t L = value_len(fs, e, any_ctrl, ctrl_s, S);
                if (L) atomicAdd(&S.rel_len[col], L);
              }
              atomicMax(&S.n_rel, col + 1);
            }
            if (isrd) { S.rd0_pos = e + 1; S.rd0_k = col; }
          }
          return;
        }
        if (in_pass && col < n_cols) slot_s[col * nrp + (rl - lo)] = (fs << 16) | e;
        if (NS > 0 && first && !emit && !defer && col < n_cols && ((P.strmask >> col) & 1u)) {
          const uint32_t L = value_len(fs, e, any_ctrl, ctrl_s, S);
          if (L) add16(cnt, P.stridx[col], L);
        }
        if (isrd && !open && col != n_cols - 1) {
          if (first && !emit && !infer) report(P.st, PP_ERR_COLCOUNT, tile_base + e, true);
          if (first && status) atomicOr(&flags_s[rl >> 5], 1u << (rl & 31u));
          if (in_pass)  // missing fields take the column default
            for (uint32_t c = col + 1; c < n_cols; ++c) slot_s[c * nrp + (rl - lo)] = SLOT_DEFAULT;
        }
      };
      // The fields of the lane's chunk in input order, each passed to
      // act(row, column (row 0: index), start, end, ends a record, still
      // open): a lane per chunk walks its terminators.  (A lane per field,
      // from a list of the warp's terminators, was measured 1-3 % slower:
      // fields spread evenly enough over the chunks.)
      auto walk = [&](auto&& act) {
        {
          uint32_t term = term_all, col = col0, rl = rl0, fs = fs0;
          bool vrd = virt_rd;
          for (;;) {
            uint32_t e;
            bool isrd;
            if (term) {
              const uint32_t j = __ffs(term) - 1;
              term &= term - 1;
              e = cstart + j;
              isrd = (rd >> j) & 1u;
            } else if (vrd) {
              e = tile_len;
              isrd = true;
              vrd = false;
            } else {
              break;
            }
            act(rl, col, fs, e, isrd, false);
            if (isrd) { ++rl; col = 0; }
            else col = col < 0x7FFFFF00u ? col + 1 : col;
            fs = e + 1;
          }
          if (owns_tail && !any_virt) act(rl, col, fs, tile_len, false, true);
        }
      };
      walk(enter);
      if (NS > 0 && first && !emit && !defer) {  // warp sums of the packed counters -> tile totals
        bool any = false;
#pragma unroll
        for (int k = 0; k < NSW; ++k) any |= cnt[k] != 0;
        if (__any_sync(FULL, any)) {
#pragma unroll
          for (int k = 0; k < NSW; ++k) {
            uint64_t v = cnt[k];
#pragma unroll
            for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
            if (lane < 4 && 4 * k + lane < int(n_str)) {
              const uint32_t x = uint32_t(v >> (16 * lane)) & 0xFFFFu;
              if (x) atomicAdd(&S.ctot[4 * k + lane], x);
            }
          }
        }
      }
      if (first) {
        if (NS > 0 && pend) {  // the previous tile's write-out, its chars offsets known
          bar_sync(BAR_CHR, NT + 32);
          write_out(0u, S.pd_rows, S.pd_rows, S.pd_rec0, S.pd_col_in, S.pd_col_end);
          pend = false;
        }
        if (NS > 0 && !emit && !defer) bar_arrive(BAR_W2, NT + 32);
        // ---- the tile's context from the look-back
        bar_sync(BAR_V2, NTF);
        rec0 = S.rec0;
        X.tile_fstart = S.last1;
        X.tile_fstate = S.last1 ? (S.lst & 0xFFu) : uint32_t(P.start_state);
        col_in = S.col_in;
        {
          const uint32_t ac = S.agg_col;
          if (ac & ABS32) {
            col_end = ac & ~ABS32;
          } else {
            const uint64_t c = uint64_t(col_in) + ac;
            col_end = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
          }
          if (any_virt) col_end = n_cols;
        }
        if (emit) {
          // dropped records known: the emitted value bytes per string
          // column, and the column-count check of every record closed here
          // that is not on the skip list
          walk([&](uint32_t rl, uint32_t col, uint32_t fs, uint32_t e, bool isrd, bool open) {
            const uint64_t rec = rec0 + rl;
            if (rl > 0 && isrd && !open && col != n_cols - 1 && !rec_skip_listed(P, rec))
              report(P.st, PP_ERR_COLCOUNT, tile_base + e, true);
            const uint32_t c = rl == 0 ? col_in + col : col;
            if (NS > 0 && c < n_cols && ((P.strmask >> c) & 1u) && !rec_dropped(P, rec)) {
              const uint32_t L = value_len(fs, e, any_ctrl, ctrl_s, S);
              if (L) atomicAdd(&S.ctot[P.stridx[c]], L);
            }
          });
          if (NS > 0) bar_arrive(BAR_W2, NT + 32);
        }
        // row 0: its fields' columns follow the entry column
        const uint32_t nrel = S.n_rel;
        if (uint32_t(t) < nrel && col_in + t < n_cols) slot_s[(col_in + t) * nrp] = S.rel_slot[t];
        if (S.rd0_pos) {
          const uint32_t nf = col_in + S.rd0_k + 1;  // fields of the record
          if (nf != n_cols) {
            if (t == 0 && !(emit && rec_skip_listed(P, rec0)) && !infer)
              report(P.st, PP_ERR_COLCOUNT, tile_base + S.rd0_pos - 1, true);
            if (t == 0 && status) atomicOr(&P.mark_bits[rec0 >> 5], 1u << (rec0 & 31u));
            for (uint32_t c = nf + t; c < n_cols; c += NT) slot_s[c * nrp] = SLOT_DEFAULT;
          }
        }
        if (status)  // the records of rows >= 1 with a wrong field count, to the input's bitmap
          for (uint32_t q = t; q < (rows + 31) / 32; q += NT) {
            uint32_t m = flags_s[q];
            while (m) {
              const uint64_t rec = rec0 + 32u * q + uint32_t(__ffs(m) - 1);
              m &= m - 1;
              atomicOr(&P.mark_bits[rec >> 5], 1u << (rec & 31u));
            }
          }
      }
      bar_sync(BAR_W, NT);
      if (!P.has_out) {  // a sizing pass: counts only
        next_ticket(b);
        if (NS > 0 && n_str) bar_sync(BAR_CHR, NT + 32);
        break;
      }
      const uint32_t ngr = (nr + 31) / 32;

      if (NS > 0 && n_str) {
        // ---- string fields: value bytes -> chars positions (block scan
        // over the column-major items), then staging copies
        const uint32_t n_items = n_str * nr;
        const uint32_t per = (n_items + NT - 1) / NT;  // <= SLOT_CAP / NT
        const uint32_t k0 = min(n_items, uint32_t(t) * per), k1 = min(n_items, k0 + per);
        uint32_t mysum = 0;
        {
          uint32_t si = k0 / nr, r = k0 - si * nr;
          for (uint32_t k = k0; k < k1; ++k) {
            uint32_t len = 0;
            const uint32_t c = P.strcol[si];
            const uint32_t row = lo + r;
            const bool closed = (row > 0 || c >= col_in) && (row + 1 < rows || c < col_end);
            const bool open = row + 1 == rows && c == col_end && !any_virt;
            if ((closed || open) && !(emit && rec_dropped(P, rec0 + row))) {
              const uint32_t v = slot_s[c * nrp + r];
              if (v != SLOT_DEFAULT) {
                const bool before = (v >> 16) == REL_START;
                const uint32_t a0 = before ? 0u : (v >> 16), e = v & 0xFFFFu;
                len = value_len(v >> 16, e, any_ctrl, ctrl_s, S);
                if (len > SHORT_FIELD) {  // mark the chunks of a long field
                  const uint32_t c0 = a0 >> 5, c1 = (e - 1) >> 5;
                  S.lk[before ? 0 : 1][c0] = uint16_t(k);
                  for (uint32_t cc = c0 + 1; cc <= c1; ++cc) S.lk[0][cc] = uint16_t(k);
                }
              }
            }
            pos_s[k] = uint16_t(len);
            mysum += len;
            if (++r == nr) { r = 0; ++si; }
          }
        }
        uint32_t xi = mysum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(FULL, xi, d);
          if (lane >= d) xi += o;
        }
        if (lane == 31) S.wsum[warp] = xi;
        bar_sync(BAR_W, NT);
        {  // lengths -> chars end positions (inclusive prefix); every warp
           // sums the warps before it itself
          const uint32_t before = __reduce_add_sync(FULL, lane < warp ? S.wsum[lane] : 0u);
          if (warp == NW - 1 && lane == 31) S.cstart[n_str] = before + xi;
          uint32_t run = before + xi - mysum;
          uint32_t si = k0 / nr, r = k0 - si * nr;
          for (uint32_t k = k0; k < k1; ++k) {
            if (r == 0) S.cstart[si] = run;
            run += pos_s[k];
            pos_s[k] = uint16_t(run);
            if (++r == nr) { r = 0; ++si; }
          }
        }
        bar_sync(BAR_W, NT);
        if (defer) bar_arrive(BAR_W2, NT + 32);  // the column totals (S.cstart) for the chars warp
        // staging: a lane per short field; long fields chunk-parallel, each
        // thread copying its chunk's part of the (at most two) long fields
        // that cover it
        {
          uint32_t si = k0 / nr, r = k0 - si * nr;
          uint32_t prev = k0 ? pos_s[k0 - 1] : 0u;
          if (r == 0) prev = S.cstart[si];
          for (uint32_t k = k0; k < k1; ++k) {
            const uint32_t pe = pos_s[k];
            const uint32_t len = pe - prev;
            prev = pe;
            const uint32_t c = P.strcol[si];
            const uint32_t rr = r;
            if (++r == nr) { r = 0; ++si; prev = si < n_str ? S.cstart[si] : prev; }
            if (len == 0 || len > SHORT_FIELD) continue;
            const uint32_t v = slot_s[c * nrp + rr];
            const uint32_t a0 = (v >> 16) == REL_START ? 0u : (v >> 16), e = v & 0xFFFFu;
            uint32_t dst = pe - len;
            if (len == e - a0) {
              for (uint32_t p = a0; p < e; ++p) stage_s[dst++] = tile_s[p];
            } else {
              for (uint32_t p = a0; p < e; ++p)
                if (!((ctrl_s[p >> 5] >> (p & 31)) & 1u)) stage_s[dst++] = tile_s[p];
            }
          }
        }
        {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t k = S.lk[h][t];
            if (k == NO_FIELD) continue;
            const uint32_t ksi = k / nr;
            const uint32_t v = slot_s[P.strcol[ksi] * nrp + (k - ksi * nr)];
            const uint32_t a0 = (v >> 16) == REL_START ? 0u : (v >> 16), e = v & 0xFFFFu;
            const uint32_t p0 = max(a0, cstart), p1 = min(e, cstart + clen);
            const uint32_t c_a0 = any_ctrl ? ctrl_bef(ctrl_s, S, a0) : 0u;
            const uint32_t c_e = any_ctrl ? ctrl_bef(ctrl_s, S, e) : 0u;
            const uint32_t c_p0 = any_ctrl ? ctrl_bef(ctrl_s, S, p0) : 0u;
            const uint32_t len = (e - a0) - (c_e - c_a0);
            uint32_t dst = pos_s[k] - len + (p0 - a0) - (c_p0 - c_a0);
            const uint32_t cm = g.ctrl & range_mask(p0 - cstart, p1 - cstart);
            // the runs between control bytes
            uint32_t q = p0, mm = cm;
            while (q < p1) {
              const uint32_t nx = mm ? cstart + uint32_t(__ffs(mm)) - 1u : p1;  // next control byte
              if (nx > q) {
                copy_run(stage_s, dst, tile_s, raw_w, toff, q, nx - q);
                dst += nx - q;
              }
              if (!mm) break;
              mm &= mm - 1u;
              q = nx + 1u;
            }
          }
        }
      }

      // ---- numbers: a lane per (numeric column, row) slot, the slots of
      // the numeric columns taken column by column, 32 to a warp; columns of
      // one type are adjacent, so a warp mostly runs one conversion
      {
        const uint32_t n_slots = S.n_num * nr;
        const uint32_t magic = nr > 1 ? 0xFFFFFFFFu / nr + 1u : 0u;  // k / nr, exact for k < 2^13
        for (uint32_t k = uint32_t(warp) * 32 + uint32_t(lane); k < n_slots; k += NT) {
          const uint32_t oc = nr > 1 ? __umulhi(k, magic) : k;
          const uint32_t c = S.numcol[oc];
          const uint32_t r = lo + (k - oc * nr);
          const uint32_t r_first = c < col_in ? 1u : 0u;  // rows whose field c closes here
          const uint32_t r_end = c < col_end ? rows : rows - 1u;
          if (r < r_first || r >= r_end) continue;
          uint64_t rec = rec0 + r;
          if (emit) {
            if (rec_dropped(P, rec)) continue;
            rec -= dropped_before(P, rec);
          }
          if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
          const uint32_t v = slot_s[c * nrp + (r - lo)];
          const uint32_t ty = S.coltype[c];
          if ((v & 0xFFFFu) - (v >> 16) > LONG_NUM) {  // (wraps for REL_START and SLOT_DEFAULT)
            // a long field goes to a warp (the queue permitting); so does,
            // with an encoding, a field begun in an earlier tile (its bytes
            // before the tile need symbol decoding)
            const uint32_t fsr = v >> 16, fe = v & 0xFFFFu;
            const uint64_t span = fsr == REL_START ? X.tile_base + fe - X.tile_fstart : fe - fsr;
            if (GEN && P.enc && v != SLOT_DEFAULT && fsr == REL_START) {
              const uint32_t q = atomicAdd(&P.s.counters[5], 1u);  // at most one per tile
              P.s.long_q[P.s.long_cap + q] = ppi::LongField{rec, X.tile_fstart, X.tile_base + fe,
                                                            c | (ty << 8),
                                                            ppi::LONG_STATE | X.tile_fstate};
              continue;
            }
            if (v != SLOT_DEFAULT && span > LONG_NUM && ty != PP_COL_TIMESTAMP &&
                ty != ppi::COL_INFER && P.s.long_q) {
              const uint32_t q = atomicAdd(&P.s.counters[4], 1u);
              if (q < P.s.long_cap) {
                P.s.long_q[q] = fsr == REL_START
                    ? ppi::LongField{rec, X.tile_fstart, X.tile_base + fe, c | (ty << 8),
                                     ppi::LONG_STATE | X.tile_fstate}
                    : ppi::LongField{rec, X.tile_base + fsr, X.tile_base + fe, c | (ty << 8), 0u};
                continue;
              }
            }
          }
          void* const out = P.typed[c];
          const uint64_t dflt = P.defval[c];
          switch (ty) {
            case PP_COL_FLOAT64: convert_store<PP_COL_FLOAT64>(P, X, out, rec, v, dflt); break;
            case PP_COL_INT64: convert_store<PP_COL_INT64>(P, X, out, rec, v, dflt); break;
            case PP_COL_TIMESTAMP: convert_store<PP_COL_TIMESTAMP>(P, X, out, rec, v, dflt); break;
            case PP_COL_INT32: convert_store<PP_COL_INT32>(P, X, out, rec, v, dflt); break;
            case ppi::COL_INFER: {
              if constexpr (GEN) {
                const uint32_t code = infer_field(P, v, X);
                if (code) atomicMax(&S.inf[c], code);
              }
              break;
            }
            default: convert_store<PP_COL_INT8>(P, X, out, rec, v, dflt); break;
          }
        }
      }
      if (first) next_ticket(b);
      bar_sync(BAR_W, NT);
      if (NS > 0 && n_str) {
        if (defer) {  // written during the next tile, once its fields are walked
          if (t == 0) { S.pd_rec0 = rec0; S.pd_rows = rows; S.pd_col_in = col_in; S.pd_col_end = col_end; }
          pend = true;
        } else {
          if (first) bar_sync(BAR_CHR, NT + 32);  // the tile's chars offsets
          write_out(lo, hi, rows, rec0, col_in, col_end);
          bar_sync(BAR_W, NT);
          if (t < int(n_str)) S.carry[t] += S.cstart[t + 1] - S.cstart[t];
        }
      }
      bar_sync(BAR_W, NT);
    }
    if (t < int(n_str)) S.carry[t] = 0;
    if (infer && t < int(n_cols) && S.inf[t]) {  // this tile's types, to the input's
      atomicMax(&P.infer_out[t], S.inf[t]);
      S.inf[t] = 0;
    }
    if (owns_end) {
      const uint64_t total = rec0 + (rows - 1) + (virt_rd ? 1u : 0u);  // records of the input
      const uint64_t dropped = emit ? dropped_before(P, total) : 0ull;
      P.st->n_records = total - dropped;
      P.st->n_dropped = dropped;
    }
    bar_sync(BAR_W, NT);
  }
}

// ===================================================== column-count inference
// ParPaRaw Section 4, "Inferring or validating number of columns": over a
// byte range, the field delimiters before its first record delimiter (all
// of them if it has none), those after its last, and the fewest and most
// fields of the records lying wholly inside it.  Ranges combine in input
// order: the records that span the seam have a.post + b.pre + 1 fields.
struct FAgg { uint32_t rd, pre, post, mn, mx; };

__device__ __forceinline__ FAgg fagg_identity() { return {0u, 0u, 0u, 0xFFFFFFFFu, 0u}; }
__device__ __forceinline__ uint32_t sat_add(uint32_t a, uint32_t b) {
  const uint32_t c = a + b;
  return c < a ? 0xFFFFFFFFu : c;
}
__device__ __forceinline__ FAgg fagg_combine(const FAgg& a, const FAgg& b) {
  if (!a.rd && !b.rd) {
    const uint32_t f = sat_add(a.pre, b.pre);
    return {0u, f, f, 0xFFFFFFFFu, 0u};
  }
  if (!a.rd) return {b.rd, sat_add(a.pre, b.pre), b.post, b.mn, b.mx};
  if (!b.rd) return {a.rd, a.pre, sat_add(a.post, b.pre), a.mn, a.mx};
  const uint32_t mid = sat_add(sat_add(a.post, b.pre), 1u);
  return {sat_add(a.rd, b.rd), a.pre, b.post, min(min(a.mn, b.mn), mid),
          max(max(a.mx, b.mx), mid)};
}
// one 32-byte chunk from its delimiter bitmaps
__device__ __forceinline__ FAgg fagg_chunk(uint32_t fd, uint32_t rd) {
  if (!rd) {
    const uint32_t f = __popc(fd);
    return {0u, f, f, 0xFFFFFFFFu, 0u};
  }
  const uint32_t first = __ffs(rd) - 1, last = 31 - __clz(rd);
  FAgg a = {uint32_t(__popc(rd)), uint32_t(__popc(fd & range_mask(0, first))),
            uint32_t(__popc(fd & range_mask(last + 1, 32))), 0xFFFFFFFFu, 0u};
  uint32_t m = rd & (rd - 1), prev = first;
  while (m) {
    const uint32_t j = __ffs(m) - 1;
    const uint32_t f = __popc(fd & range_mask(prev + 1, j)) + 1u;
    a.mn = min(a.mn, f);
    a.mx = max(a.mx, f);
    prev = j;
    m &= m - 1;
  }
  return a;
}
// ordered reduction over the warp: lane 0 gets lanes 0..31 combined in order
__device__ __forceinline__ FAgg fagg_warp(FAgg a) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const FAgg o = {__shfl_down_sync(FULL, a.rd, d), __shfl_down_sync(FULL, a.pre, d),
                    __shfl_down_sync(FULL, a.post, d), __shfl_down_sync(FULL, a.mn, d),
                    __shfl_down_sync(FULL, a.mx, d)};
    if (lane + d < 32) a = fagg_combine(a, o);
  }
  return a;
}

struct FieldsShared {
  Feed F;
  uint32_t tile_stv;
  uint32_t warp_stv[NW];
  FAgg wagg[NW];
};
constexpr size_t FIELDS_SMEM = LUT_BYTES + 2 * TILE + sizeof(FieldsShared);

// Per tile, from its true start state: tag every chunk, then the tile's
// aggregate; the thread that owns the input's last byte records whether the
// input ends inside a record (counters[2]).
__global__ void __launch_bounds__(NT, 3) fields_kernel(const __grid_constant__ ParseParams P,
                                                       FAgg* agg) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin0 = smem + LUT_BYTES;  // two tile buffers
  FieldsShared& S = *reinterpret_cast<FieldsShared*>(lin0 + 2 * TILE);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  load_lut(P, lut_s);
  const uint32_t* my_lut = lut_s + lane;
  const bool aligned_in = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;
  uint32_t* counter = &P.s.counters[0];
  uint32_t tk = 0;  // thread 0: the next ticket
  feed_start(P, S.F, counter, aligned_in, lin0, tk);
  for (;;) {
    const uint32_t tile = S.F.tile[S.F.cur];
    if (tile >= P.n_tiles) break;
    uint8_t* tile_s = lin0 + S.F.cur * TILE;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    uint32_t w[8];
    feed_tile(P, S.F, counter, aligned_in, lin0, tile_base, tile_len, w, tk);
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    const uint32_t s_tile = P.s.tile_state[tile];
    uint32_t G, special, special_x;
    stv_pass(w, clen, tile_s, cstart, my_lut, G, special, special_x);
    const uint32_t lane_ex = block_stv(G, S.warp_stv, &S.tile_stv);
    const uint32_t st = stv_apply(lane_ex, stv_apply(S.warp_stv[warp], s_tile));
    const Tags g = tag_chunk(st, special, special_x, P.sticky, clen, cstart, tile_s + cstart,
                             my_lut, P.bg_next);
    if (g.inv_at < clen && st != 4)
      report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + g.inv_at, true);
    if (tile + 1 == P.n_tiles && clen > 0 && cstart + clen == tile_len) {
      if (g.end != 4 && !((P.accept_mask >> g.end) & 1u)) report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
      P.s.counters[2] = ((g.rd >> (clen - 1)) & 1u) ? 0u : 1u;
    }
    const FAgg a = fagg_warp(fagg_chunk(g.fd, g.rd));
    if (lane == 0) S.wagg[warp] = a;
    __syncthreads();
    if (warp == 0) {
      const FAgg b = fagg_warp(lane < NW ? S.wagg[lane] : fagg_identity());
      if (lane == 0) agg[tile] = b;
    }
    feed_next(S.F);  // the tile was last read before the barrier above
  }
  feed_finish(S.F);
}

// The tiles' aggregates in input order (one block), then the records at the
// input's two ends: the first record ends at the first record delimiter,
// and an open tail is one more record.
constexpr int FR_NT = 1024;
__global__ void __launch_bounds__(FR_NT) fields_reduce_kernel(const __grid_constant__ ParseParams P,
                                                              const FAgg* agg, uint64_t* out) {
  __shared__ FAgg wa[FR_NT / 32];
  __shared__ unsigned long long n_rd;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) n_rd = 0;
  __syncthreads();
  const uint32_t n = P.n_tiles, per = (n + FR_NT - 1) / FR_NT;
  const uint32_t i0 = min(n, uint32_t(t) * per), i1 = min(n, i0 + per);
  FAgg a = fagg_identity();
  unsigned long long rds = 0;
  for (uint32_t i = i0; i < i1; ++i) {
    const FAgg b = agg[i];
    a = fagg_combine(a, b);
    rds += b.rd;
  }
  if (rds) atomicAdd(&n_rd, rds);
  a = fagg_warp(a);
  if (lane == 0) wa[warp] = a;
  __syncthreads();
  if (warp == 0) {
    a = fagg_warp(wa[lane]);
    if (lane == 0) {
      const bool tail = n > 0 && P.s.counters[2] != 0;
      uint64_t mn = a.mn, mx = a.mx;
      if (a.rd) {  // the first record, up to the first record delimiter
        mn = min(mn, uint64_t(a.pre) + 1);
        mx = max(mx, uint64_t(a.pre) + 1);
        if (tail) {  // the open tail after the last one
          mn = min(mn, uint64_t(a.post) + 1);
          mx = max(mx, uint64_t(a.post) + 1);
        }
      } else if (tail) {  // one record, the whole input
        mn = mx = uint64_t(a.pre) + 1;
      }
      const uint64_t recs = n_rd + (tail ? 1u : 0u);
      out[0] = recs ? mn : 0;
      out[1] = recs ? mx : 0;
      P.st->n_records = recs;
    }
  }
}

// ================================================================= launch
// Zero the tile counters and the look-back flags; initialise the status and
// offsets[c][0] = 0 for every string column.
__global__ void parse_init_kernel(ParseParams P) {
  const ppi::ParseScratch& s = P.s;
  const uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t stride = gridDim.x * blockDim.x;
  if (s.v2_desc)
    for (uint32_t i = i0; i < P.n_tiles; i += stride) {
      s.v2_desc[2 * size_t(i)] = 0;
      s.v2_desc[2 * size_t(i) + 1] = 0;
    }
  if (s.c_flag)
    for (uint32_t i = i0; i < P.n_tiles; i += stride) s.c_flag[i] = 0;
  for (uint32_t i = i0; i < s.n_tstate_blocks; i += stride) s.tstate_words[i] = 0;
  if (i0 < 6) s.counters[i0] = 0;
  if (i0 == 0) {
    pp_status* st = P.st;
    st->error = 0;
    st->reserved = 0;
    st->first_error_offset = ~0ull;
    st->n_records = 0;
    st->n_tokens = 0;
    for (int c = 0; c < PP_MAX_COLS; ++c) st->chars_len[c] = 0;
    st->n_dropped = 0;
    if (P.has_out)
      for (int c = 0; c < P.n_str; ++c) P.offsets[c][0] = 0;
  }
}

uint32_t init_grid(uint32_t n) {
  return std::max<uint32_t>(1, std::min<uint32_t>((n + 255) / 256, 1024));
}

// Per device: the SM count, the tile pass's dynamic shared-memory attribute
// and its resident blocks per SM.
struct Occ { int blocks = 1, n_sm = 0, tv_blocks = 1; };  // tile pass and tile-vector blocks per SM

template <int NS, bool GEN>
cudaError_t parse_setup(Occ** out) {
  static ppi::DeviceOnce once;
  static Occ occ[ppi::MAX_DEVICES];
  int dev;
  cudaError_t e = ppi::current_device(&dev);
  if (e != cudaSuccess) return e;
  e = once.run(dev, [](int d) {
    Occ o;
    cudaError_t r;
    if ((r = ppi::sm_count(&o.n_sm)) != cudaSuccess) return r;
    if ((r = cudaFuncSetAttribute(parse_kernel<NS, GEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(PARSE_SMEM))) != cudaSuccess)
      return r;
    int b = 0;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, parse_kernel<NS, GEN>, ntf_of<NS>(),
                                                           PARSE_SMEM)) != cudaSuccess)
      return r;
    o.blocks = b > 0 ? b : 1;
    // the tile-vector pass: a grid of exactly the resident blocks (a second,
    // partial wave would leave most SMs idle at its end)
    if ((r = cudaFuncSetAttribute(tile_stv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  TV_SMEM)) != cudaSuccess)
      return r;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, tile_stv_kernel, TV_NT,
                                                           TV_SMEM)) != cudaSuccess)
      return r;
    o.tv_blocks = b > 0 ? b : 1;
    occ[d] = o;
    return cudaSuccess;
  });
  *out = &occ[dev];
  return e;
}

template <int NS, bool GEN>
cudaError_t launch_ns(const ParseParams& p, cudaStream_t stream) {
  Occ* po = nullptr;
  cudaError_t e = parse_setup<NS, GEN>(&po);
  if (e != cudaSuccess) return e;
  const Occ& occ = *po;
  const bool timed = ppi::stage_begin();
  if (timed) ppi::stage_mark(0, stream);
  parse_init_kernel<<<init_grid(std::max(p.n_tiles, p.s.n_tstate_blocks)), 256, 0, stream>>>(p);
  if (timed) ppi::stage_mark(1, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) {
    const uint32_t gv = uint32_t(std::min<uint64_t>((p.n_tiles + TV_NT / 32 - 1) / (TV_NT / 32),
                                                    uint64_t(occ.n_sm) * occ.tv_blocks));
    tile_stv_kernel<<<gv, TV_NT, TV_SMEM, stream>>>(p);
  }
  if (timed) ppi::stage_mark(2, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) tile_state_kernel<<<p.s.n_tstate_blocks, TS_NT, 0, stream>>>(p);
  if (timed) ppi::stage_mark(3, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const uint32_t g = uint32_t(std::min<uint64_t>(std::max<uint32_t>(p.n_tiles, 1),
                                                 uint64_t(occ.n_sm) * occ.blocks));
  if (p.n_tiles) parse_kernel<NS, GEN><<<g, ntf_of<NS>(), PARSE_SMEM, stream>>>(p);
  if (timed) ppi::stage_mark(4, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the long numeric fields the tile pass queued (an empty queue costs a
  // launch that returns at once)
  bool any_num = false;
  for (int c = 0; c < p.n_cols; ++c)
    any_num |= p.coltype[c] == PP_COL_INT8 || p.coltype[c] == PP_COL_INT32 ||
               p.coltype[c] == PP_COL_INT64 || p.coltype[c] == PP_COL_FLOAT64;
  if (p.n_tiles && p.has_out && any_num && p.s.long_q)
    long_field_kernel<<<std::max(1, occ.n_sm), LF_NT, 0, stream>>>(p);
  if (timed) ppi::stage_mark(5, stream);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cudaError_t launch_fields(const ParseParams& p, FAgg* agg, uint64_t* out, cudaStream_t stream) {
  static ppi::DeviceOnce once;
  static int occ_of[ppi::MAX_DEVICES];
  int dev, n_sm = 0;
  cudaError_t e;
  if ((e = ppi::current_device(&dev)) != cudaSuccess) return e;
  if ((e = ppi::sm_count(&n_sm)) != cudaSuccess) return e;
  e = once.run(dev, [](int d) {
    cudaError_t r = cudaFuncSetAttribute(fields_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(FIELDS_SMEM));
    if (r != cudaSuccess) return r;
    if ((r = cudaFuncSetAttribute(tile_stv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  TV_SMEM)) != cudaSuccess)
      return r;
    int b = 0;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fields_kernel, NT, FIELDS_SMEM)) !=
        cudaSuccess)
      return r;
    occ_of[d] = b > 0 ? b : 1;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int occ = occ_of[dev];
  parse_init_kernel<<<init_grid(p.s.n_tstate_blocks), 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) {
    const uint32_t gv = uint32_t(std::min<uint64_t>((p.n_tiles + TV_NT / 32 - 1) / (TV_NT / 32),
                                                    uint64_t(n_sm) * 3));
    tile_stv_kernel<<<gv, TV_NT, TV_SMEM, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    tile_state_kernel<<<p.s.n_tstate_blocks, TS_NT, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const uint32_t g = uint32_t(std::min<uint64_t>(p.n_tiles, uint64_t(n_sm) * occ));
    fields_kernel<<<g, NT, FIELDS_SMEM, stream>>>(p, agg);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  fields_reduce_kernel<<<1, FR_NT, 0, stream>>>(p, agg, out);
  return cudaGetLastError();
}

}  // namespace

namespace ppi {

size_t parse_tile_bytes() { return TILE; }

// counters | tile vectors | tile states | tile-state look-back words | tile aggregates
size_t fields_scratch_bytes(uint32_t n) {
  const uint32_t nt = (n + TS_TILES - 1) / TS_TILES;
  return 256 + align256(size_t(n) * 4) + align256(n) + align256(size_t(nt) * 8) +
         align256(size_t(n) * sizeof(FAgg));
}

cudaError_t launch_count_fields(ParseParams p, void* scratch, uint64_t* out, cudaStream_t stream) {
  uint8_t* b = static_cast<uint8_t*>(scratch);
  const uint32_t n = p.n_tiles;
  p.s = ParseScratch{};
  p.s.counters = reinterpret_cast<uint32_t*>(b); b += 256;
  p.s.tile_stv = reinterpret_cast<uint32_t*>(b); b += align256(size_t(n) * 4);
  p.s.tile_state = b; b += align256(n);
  p.s.n_tstate_blocks = (n + TS_TILES - 1) / TS_TILES;
  p.s.tstate_words = reinterpret_cast<unsigned long long*>(b);
  b += align256(size_t(p.s.n_tstate_blocks) * 8);
  return launch_fields(p, reinterpret_cast<FAgg*>(b), out, stream);
}

cudaError_t launch_infer_finish(const uint32_t* codes, int32_t* types, int n, cudaStream_t stream) {
  infer_finish_kernel<<<1, 64, 0, stream>>>(codes, types, n);
  return cudaGetLastError();
}

int parse_ns_width(int n_str) {
  if (n_str <= 0) return 0;
  if (n_str <= 4) return 4;
  if (n_str <= 8) return 8;
  return 16;
}

// layout: counters | tile vectors | tile states | tile-state look-back words |
// context look-back descriptors (16 bytes a tile) | chars look-back (flags,
// aggregates, inclusive prefixes: ns words a tile)
// Long numeric fields queued per call: a tile starts at most TILE / LONG_NUM
// of them, plus the one open at its start.
uint32_t long_cap(uint32_t n) {
  return uint32_t(std::min<uint64_t>(ppi::LONG_CAP, uint64_t(n) * (TILE / LONG_NUM + 1)));
}

size_t parse_scratch_bytes(uint32_t n, int ns, bool sym) {
  const uint32_t nt = (n + TS_TILES - 1) / TS_TILES;
  const int k3 = ns > 0 ? ns : 1;
  const size_t nq = size_t(long_cap(n)) + (sym ? n : 0u);
  return 256 + align256(size_t(n) * 4) + align256(n) + align256(size_t(nt) * 8) +
         align256(size_t(n) * 16) + align256(nq * sizeof(ppi::LongField)) +
         (ns > 0 ? align256(size_t(n) * 4) + 2 * align256(size_t(n) * k3 * 8) : 0);
}

void parse_scratch_carve(void* base, uint32_t n, int ns, ParseScratch* o, bool sym) {
  const int k3 = ns > 0 ? ns : 1;
  uint8_t* p = static_cast<uint8_t*>(base);
  *o = ParseScratch{};
  o->counters = reinterpret_cast<uint32_t*>(p); p += 256;
  o->tile_stv = reinterpret_cast<uint32_t*>(p); p += align256(size_t(n) * 4);
  o->tile_state = p; p += align256(n);
  o->n_tstate_blocks = (n + TS_TILES - 1) / TS_TILES;
  o->tstate_words = reinterpret_cast<unsigned long long*>(p);
  p += align256(size_t(o->n_tstate_blocks) * 8);
  o->v2_desc = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 16);
  o->long_cap = long_cap(n);
  o->long_q = reinterpret_cast<ppi::LongField*>(p);
  p += align256((size_t(o->long_cap) + (sym ? n : 0u)) * sizeof(ppi::LongField));
  if (ns > 0) {
    o->c_flag = reinterpret_cast<uint32_t*>(p); p += align256(size_t(n) * 4);
    o->c_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * k3 * 8);
    o->c_inc = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * k3 * 8);
  }
}

cudaError_t launch_parse(const ParseParams& p, cudaStream_t stream) {
  // the general kernel for encodings, the options, type inference and
  // streamed chunks
  const bool gen = p.enc || p.drop_bits || p.mark_bits || p.infer_out || p.record_end ||
                   p.dbg_tags;
  switch (parse_ns_width(p.n_str)) {
    case 0: return gen ? launch_ns<0, true>(p, stream) : launch_ns<0, false>(p, stream);
    case 4: return gen ? launch_ns<4, true>(p, stream) : launch_ns<4, false>(p, stream);
    case 8: return gen ? launch_ns<8, true>(p, stream) : launch_ns<8, false>(p, stream);
    default: return gen ? launch_ns<16, true>(p, stream) : launch_ns<16, false>(p, stream);
  }
}

}  // namespace ppi

extern "C" pp_rc pp_debug_long_fields(uint64_t* out, int reset) {
  unsigned long long v = 0;
  if (out && cudaMemcpyFromSymbol(&v, g_long_fields, sizeof(v)) != cudaSuccess) return PP_ECUDA;
  if (out) *out = v;
  if (reset) {
    v = 0;
    if (cudaMemcpyToSymbol(g_long_fields, &v, sizeof(v)) != cudaSuccess) return PP_ECUDA;
  }
  return PP_OK;
}
