// pp_parse: DFA-based parsing of delimiter-separated input into Arrow-style
// columns on sm_103a, in three kernels with no inter-tile waiting on the hot
// path.
//
// The input is cut into 16 KiB tiles; each tile is one CTA of 512 threads
// and each thread owns a 32-byte chunk (one bit per byte in the bitmap
// indexes).  Tiles reach shared memory by a 1-D bulk copy (TMA engine)
// into one of two linear buffers, the next tile landing in the other while
// the current one is processed.
//
// 1. Context pass (ctx_kernel).  Each thread runs the multi-instance DFA
//    over its chunk (ParPaRaw Section 3.1, Figure 2): the transition vector
//    of the four live states sits in one register, one byte per state, and
//    each byte composes it with its symbol group's row by one byte-permute
//    (the row-per-group transition table of ParPaRaw Section 5, Table 1,
//    read from a per-lane replicated shared-memory LUT).  Vectors compose
//    across the warp (shuffles) and the block.  Because the tile's true
//    start state is not known yet, the tile then tags its bytes once per
//    possible start state (threads whose start state does not depend on it
//    tag once) and records, per start state: record count, absolute or
//    relative column offset (ParPaRaw Section 3.2, Figure 4), last
//    terminator, value bytes per string column for fields whose column is
//    known inside the tile, and value bytes per relative field of the
//    tile's first, partial record.
// 2. Scan (scan_kernel).  An exclusive scan over tiles with the composite
//    operation on transition vectors (ParPaRaw Section 3.1) and the
//    record-count / column-offset operators (Section 3.2), each applied per
//    start state, resolves every tile's true start state, record index,
//    column and last terminator; the tile's value bytes per string column
//    then follow from its column, and a second scan turns them into chars
//    offsets.  Blocks chain by a single-pass decoupled look-back.
// 3. Main pass (main_kernel).  With its context known, each tile tags its
//    bytes (re-running one DFA per thread over the non-background bytes
//    only), scans record and column indices across the block, compacts
//    string value bytes per column into shared memory (stream compaction in
//    place of ParPaRaw's radix partitioning, Section 3.3) and writes them as
//    16-byte stores, and enters every closed field in a column-major
//    (column, record) slot table; one lane per field then writes the Arrow
//    offset or converts the number (Section 3.3), so a warp handles one
//    column, one type, with coalesced stores.
#include <cstdint>
#include <cuda_runtime.h>
#include <algorithm>

#include "pp.h"
#include "pp_device.cuh"
#include "pp_internal.h"
#include "pp_numeric.cuh"

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
constexpr uint32_t SLOT_ABSENT = 0xFFFFFFFEu;  // field not closed in this tile
constexpr uint32_t SLOT_DEFAULT = 0xFFFFFFFDu; // missing field: column default
constexpr uint32_t WAIT_LIMIT = 1u << 24;      // bounded mbarrier polls
constexpr int SCAN_NT = 256;           // scan kernel threads
constexpr int SCAN_TPT = 8;            // tiles per scan thread
constexpr int SCAN_TILES = SCAN_NT * SCAN_TPT;
constexpr int CTX_HDR = 52;            // stv + rec[4] + col[4] + last[4]

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

// ------------------------------------------------- tile feeding (TMA)
// Two linear landing buffers: while a tile is processed from one, the next
// tile's bulk copy lands in the other.
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

__device__ __forceinline__ void feed_start(const ParseParams& P, Feed& F, uint32_t* counter,
                                           bool aligned_in, uint8_t* lin0) {
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&F.bar[b], 1);
      F.parity[b] = 0;
      F.tile[b] = atomicAdd(counter, 1u);
      F.issued[b] = issue_tile(P, F.tile[b], aligned_in, lin0 + b * TILE, &F.bar[b]);
    }
    F.cur = 0;
  }
  __syncthreads();
}

// Wait until the current tile is in its landing buffer (plain loads for a
// ragged tail or unaligned input) and load this thread's chunk words.
__device__ __forceinline__ void feed_tile(const ParseParams& P, Feed& F, uint8_t* lin_s,
                                          uint64_t tile_base, uint32_t tile_len, uint32_t (&w)[8]) {
  const int t = threadIdx.x;
  const uint32_t b = F.cur;
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
  const uint4* src = reinterpret_cast<const uint4*>(lin_s + uint32_t(t) * CB);
  const int sw = (t >> 2) & 1;  // alternate read order: conflict-free 16-byte reads
  const uint4 x = src[sw], y = src[sw ^ 1];
  const uint4 lo = sw ? y : x, hi = sw ? x : y;
  w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
  w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
}

// After the last read of the current buffer (behind a block barrier):
// refill it with the next tile and switch buffers.
__device__ __forceinline__ void feed_next(const ParseParams& P, Feed& F, uint32_t* counter,
                                          bool aligned_in, uint8_t* lin0) {
  if (threadIdx.x == 0) {
    const uint32_t b = F.cur;
    if (F.issued[b]) F.parity[b] ^= 1u;
    F.tile[b] = atomicAdd(counter, 1u);
    F.issued[b] = issue_tile(P, F.tile[b], aligned_in, lin0 + b * TILE, &F.bar[b]);
    F.cur = b ^ 1u;
  }
  __syncthreads();
}

__device__ __forceinline__ void feed_finish(Feed& F) {
  // never leave with a bulk copy in flight into this CTA's shared memory
  if (threadIdx.x == 0)
    for (int b = 0; b < 2; ++b)
      if (F.issued[b]) mbar_wait_bounded(&F.bar[b], F.parity[b], WAIT_LIMIT);
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
// re-tagged by running the DFA from the state at its first byte.
template <class Acc>
__device__ __forceinline__ uint32_t feed_field(Acc& acc, const uint8_t* in, uint64_t fs,
                                               uint64_t fe, uint64_t tile_base,
                                               const uint8_t* tile_s, const uint32_t* ctrl_s,
                                               const uint32_t* my_lut, uint32_t fstate) {
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
                                        : uint32_t(__ldg(in + p));
      const uint32_t e = my_lut[b << 5];
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
// 8 bytes of the tile from position p (little-endian: byte p lowest); bytes
// past the tile are unspecified but stay inside shared memory.
__device__ __forceinline__ uint64_t tile_load8(const uint32_t* tile_w, uint32_t p) {
  const uint32_t q = p >> 2, sh = (p & 3u) * 8u;
  const uint32_t w0 = tile_word(tile_w, q), w1 = tile_word(tile_w, q + 1),
                 w2 = tile_word(tile_w, q + 2);
  return uint64_t(__funnelshift_r(w0, w1, sh)) | (uint64_t(__funnelshift_r(w1, w2, sh)) << 32);
}

// Copy the chunk's bytes selected by `seg` (runs of set bits) from the tile
// to stage_s from dst on.
__device__ __forceinline__ void stage_runs(uint32_t seg, uint32_t dst, const uint8_t* chunk,
                                           uint8_t* stage_s) {
  for (uint32_t m = seg; m; m &= m - 1) stage_s[dst++] = chunk[__ffs(m) - 1];
}

// ------------------------------------------------- numeric fast paths
// Digit values of the low n bytes of x (1 <= n <= 8) left-aligned for the
// combining steps, or false if one of them is not a digit.
__device__ __forceinline__ bool swar_digits(uint64_t x, uint32_t n, uint64_t& d) {
  const uint64_t keep = n >= 8 ? ~0ull : ((1ull << (8 * n)) - 1);
  x &= keep;
  const uint64_t hiok = (x & (0xF0F0F0F0F0F0F0F0ull & keep)) ^ (0x3030303030303030ull & keep);
  const uint64_t lo = x & 0x0F0F0F0F0F0F0F0Full;
  const uint64_t big = (lo + 0x0606060606060606ull) & 0xF0F0F0F0F0F0F0F0ull;
  if (hiok | big) return false;
  d = n >= 8 ? lo : lo << (8 * (8 - n));
  return true;
}
// value of 8 left-aligned digits, most significant in the lowest byte
__device__ __forceinline__ uint64_t swar_value(uint64_t d) {
  d = (d * 10 + (d >> 8)) & 0x00FF00FF00FF00FFull;
  d = (d * 100 + (d >> 16)) & 0x0000FFFF0000FFFFull;
  return (d * 10000 + (d >> 32)) & 0xFFFFFFFFull;
}
// Plain [+-]?[0-9]{1,16} field [a, a+L) of the tile: magnitude and sign.
__device__ __forceinline__ bool fast_int(const uint32_t* tile_w, uint32_t a, uint32_t L, uint64_t& mag,
                                         bool& neg) {
  uint64_t x = tile_load8(tile_w, a);
  const uint32_t c0 = uint32_t(x & 0xFFu);
  neg = c0 == '-';
  uint32_t skip = (c0 == '-' || c0 == '+') ? 1u : 0u;
  const uint32_t n = L - skip;
  if (n == 0 || n > 16) return false;
  if (skip) x = tile_load8(tile_w, a + 1);
  uint64_t d;
  if (n <= 8) {
    if (!swar_digits(x, n, d)) return false;
    mag = swar_value(d);
    return true;
  }
  if (!swar_digits(x, 8, d)) return false;
  const uint64_t hi = swar_value(d);
  uint64_t d2;
  if (!swar_digits(tile_load8(tile_w, a + skip + 8), n - 8, d2)) return false;
  const uint32_t m = n - 8;
  uint64_t p10 = 1;
  for (uint32_t i = 0; i < m; ++i) p10 *= 10;
  mag = hi * p10 + swar_value(d2);
  return true;
}
// Plain [+-]?digits[.digits] field of at most 8 characters after the sign:
// significand and decimal exponent.
__device__ __forceinline__ bool fast_float(const uint32_t* tile_w, uint32_t a, uint32_t L,
                                           uint64_t& mant, int& q, bool& neg) {
  uint64_t x = tile_load8(tile_w, a);
  const uint32_t c0 = uint32_t(x & 0xFFu);
  neg = c0 == '-';
  const uint32_t skip = (c0 == '-' || c0 == '+') ? 1u : 0u;
  const uint32_t n = L - skip;
  if (n == 0 || n > 8) return false;
  if (skip) x = (x >> 8) | (uint64_t(tile_load8(tile_w, a + 8) & 0xFFu) << 56);
  const uint64_t keep = n >= 8 ? ~0ull : ((1ull << (8 * n)) - 1);
  const uint64_t z = (x ^ 0x2E2E2E2E2E2E2E2Eull) & keep;  // zero bytes at '.'
  const uint64_t dots = ~(((z & 0x7F7F7F7F7F7F7F7Full) + 0x7F7F7F7F7F7F7F7Full) | z |
                          0x7F7F7F7F7F7F7F7Full) & keep;
  uint32_t nd = n;
  q = 0;
  if (dots) {
    if (dots & (dots - 1)) return false;                // two dots
    const uint32_t k = (__ffsll(dots) - 1) >> 3;        // dot index
    const uint64_t below = k ? ((1ull << (8 * k)) - 1) : 0ull;
    x = (x & below) | ((x >> 8) & ~below);              // squeeze the dot out
    nd = n - 1;
    q = -int(nd - k);
    if (nd == 0) return false;
  }
  uint64_t d;
  if (!swar_digits(x, nd, d)) return false;
  mant = swar_value(d);
  return true;
}

__device__ __forceinline__ void load_lut(const ParseParams& P, uint32_t* lut_s) {
  for (int k = threadIdx.x; k < 256 * 32; k += NT) lut_s[k] = P.lut[k >> 5];
}

// ================================================================ 1. context
struct CtxShared {
  Feed F;
  uint32_t tile_stv;
  uint32_t warp_stv[NW];
  uint32_t wv[NW][12];       // per warp: V2 for the four start states
  uint32_t agg[12];          // tile aggregates per start state
  uint64_t wcnt[NW][4][4];   // per warp, per state: packed string counts
  uint32_t rel[4][PP_MAX_COLS];
  int8_t stridx[PP_MAX_COLS];
};
constexpr size_t CTX_SMEM = LUT_BYTES + 2 * TILE + sizeof(CtxShared);

template <int NS>
__global__ void __launch_bounds__(NT, 2) ctx_kernel(const __grid_constant__ ParseParams P) {
  constexpr int NSW = NS > 0 ? (NS + 3) / 4 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin0 = smem + LUT_BYTES;  // two tile buffers
  CtxShared& S = *reinterpret_cast<CtxShared*>(lin0 + 2 * TILE);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  load_lut(P, lut_s);
  for (int k = t; k < PP_MAX_COLS; k += NT) S.stridx[k] = P.stridx[k];
  const uint32_t* my_lut = lut_s + lane;
  const uint32_t n_cols = uint32_t(P.n_cols);
  const bool aligned_in = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;
  uint32_t* counter = &P.s.counters[0];
  feed_start(P, S.F, counter, aligned_in, lin0);

  for (;;) {
    const uint32_t tile = S.F.tile[S.F.cur];
    if (tile >= P.n_tiles) break;
    uint8_t* tile_s = lin0 + S.F.cur * TILE;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    uint32_t w[8];
    feed_tile(P, S.F, tile_s, tile_base, tile_len, w);
    const uint32_t cstart = uint32_t(t) * CB;
    const uint8_t* own = tile_s + cstart;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    if (NS > 0)
      for (int k = t; k < 4 * PP_MAX_COLS; k += NT) (&S.rel[0][0])[k] = 0;

    uint32_t G, special, special_x;
    stv_pass(w, clen, tile_s, cstart, my_lut, G, special, special_x);
    const uint32_t lane_ex = block_stv(G, S.warp_stv, &S.tile_stv);
    const uint32_t wex = S.warp_stv[warp];

    // tag once per distinct start state of this chunk
    uint32_t st[4];
    Tags g[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      st[s] = stv_apply(lane_ex, stv_apply(wex, uint32_t(s)));
      int same = -1;
#pragma unroll
      for (int q = 0; q < s; ++q)
        if (same < 0 && st[q] == st[s]) same = q;
      if (same >= 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q == same) g[s] = g[q];
      } else {
        g[s] = tag_chunk(st[s], special, special_x, P.sticky, clen, cstart, own, my_lut,
                         P.bg_next);
      }
    }

    // block scan of (rec, col, last) for each start state
    V2 vi[4], ve[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) vi[s] = chunk_v2(g[s]);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const V2 o = shfl_up_v2(vi[s], d);
        if (lane >= d) vi[s] = op2_32(o, vi[s]);
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      ve[s] = shfl_up_v2(vi[s], 1);
      if (lane == 0) ve[s] = {0u, 0u, 0u};
    }
    if (lane == 31) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        S.wv[warp][3 * s] = vi[s].rec; S.wv[warp][3 * s + 1] = vi[s].col; S.wv[warp][3 * s + 2] = vi[s].last;
      }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        V2 x = lane < NW ? V2{S.wv[lane][3 * s], S.wv[lane][3 * s + 1], S.wv[lane][3 * s + 2]}
                         : V2{0u, 0u, 0u};
#pragma unroll
        for (int d = 1; d < NW; d <<= 1) {
          const V2 o = shfl_up_v2(x, d);
          if (lane >= d) x = op2_32(o, x);
        }
        V2 xe = shfl_up_v2(x, 1);
        if (lane == 0) xe = {0u, 0u, 0u};
        __syncwarp();
        if (lane < NW) { S.wv[lane][3 * s] = xe.rec; S.wv[lane][3 * s + 1] = xe.col; S.wv[lane][3 * s + 2] = xe.last; }
        if (lane == NW - 1) { S.agg[3 * s] = x.rec; S.agg[3 * s + 1] = x.col; S.agg[3 * s + 2] = x.last; }
      }
    }
    __syncthreads();

    // value bytes per string column: absolute columns, or relative fields
    // of the tile's first (partial) record
    uint64_t cnt[4][NSW];
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int k = 0; k < NSW; ++k) cnt[s][k] = 0;
    if (NS > 0) {
      uint32_t s_k0[4], s_n0[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const V2 pre = op2_32(V2{S.wv[warp][3 * s], S.wv[warp][3 * s + 1], S.wv[warp][3 * s + 2]}, ve[s]);
        int same = -1;
#pragma unroll
        for (int q = 0; q < s; ++q) {
          const V2 pq = op2_32(V2{S.wv[warp][3 * q], S.wv[warp][3 * q + 1], S.wv[warp][3 * q + 2]}, ve[q]);
          if (same < 0 && st[q] == st[s] && (pq.col & ABS32) && pq.col == pre.col) same = q;
        }
        if (same >= 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q == same)
#pragma unroll
              for (int k = 0; k < NSW; ++k) cnt[s][k] = cnt[q][k];
          s_k0[s] = 0xFFFFFFFFu;
          s_n0[s] = 0;
          continue;
        }
        const Tags& gs = g[s];
        const uint32_t valid = range_mask(0, min(clen, gs.inv_at));
        const uint32_t data = valid & ~(gs.fd | gs.rd | gs.ctrl);
        bool abs = (pre.col & ABS32) != 0;
        uint32_t col = pre.col & ~ABS32, term = gs.fd | gs.rd, start = 0;
        uint32_t k0 = 0xFFFFFFFFu, n0 = 0;  // first relative segment, summed per warp below
        for (;;) {
          const uint32_t j = term ? uint32_t(__ffs(term) - 1) : 32u;
          const uint32_t n = __popc(data & range_mask(start, j));
          if (n && col < n_cols) {
            if (abs) {
              const int si = S.stridx[col];
              if (si >= 0) add16(cnt[s], si, n);
            } else if (start == 0) {
              k0 = col;
              n0 = n;
            } else {
              atomicAdd(&S.rel[s][col], n);
            }
          }
          if (j == 32) break;
          if ((gs.rd >> j) & 1u) { abs = true; col = 0; }
          else col = col < 0x7FFFFF00u ? col + 1 : col;
          start = j + 1;
          term &= term - 1;
        }
        s_k0[s] = k0;
        s_n0[s] = n0;
      }
      // relative first segments: one shared atomic per (warp, field index)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t grp = __match_any_sync(FULL, s_k0[s]);
        const uint32_t sum = __reduce_add_sync(grp, s_n0[s]);
        if (s_k0[s] != 0xFFFFFFFFu && (grp & ((1u << lane) - 1)) == 0 && sum)
          atomicAdd(&S.rel[s][s_k0[s]], sum);
      }
      // block sums of the packed counters
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int k = 0; k < NSW; ++k) {
          uint64_t v = cnt[s][k];
#pragma unroll
          for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
          if (lane == 0) S.wcnt[warp][s][k] = v;
        }
    }
    __syncthreads();

    // write the tile's context record
    uint8_t* rec = P.s.ctx + size_t(tile) * P.s.ctx_stride;
    if (t < 13) {
      const uint32_t v = t == 0 ? S.tile_stv : S.agg[t - 1];
      reinterpret_cast<uint32_t*>(rec)[t] = v;
    }
    if (NS > 0) {
      uint16_t* cabs = reinterpret_cast<uint16_t*>(rec + CTX_HDR);
      uint16_t* crel = cabs + 4 * P.n_str;
      if (t < 4 * P.n_str) {
        const int s = t / P.n_str, si = t - s * P.n_str;
        uint64_t sum = 0;
        for (int q = 0; q < NW; ++q) sum += S.wcnt[q][s][si >> 2];
        cabs[t] = uint16_t((sum >> (16 * (si & 3))) & 0xFFFFu);
      }
      for (int k = t; k < 4 * int(n_cols); k += NT) {
        const int s = k / int(n_cols), c = k - s * int(n_cols);
        crel[k] = uint16_t(S.rel[s][c]);
      }
    }
    feed_next(P, S.F, counter, aligned_in, lin0);  // the tile was last read before the barrier above
  }
  feed_finish(S.F);
}

// ==================================================================== 2. scan
// Per-start-state aggregate over a run of tiles.
struct SAgg {
  uint32_t T;
  uint32_t col[4], lst[4];
  uint64_t rec[4], last1[4];
};

__device__ __forceinline__ SAgg sagg_identity(bool seed) {
  SAgg a;
  a.T = STV_ID;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    a.col[s] = seed ? ABS32 : 0u;
    a.lst[s] = 0;
    a.rec[s] = 0;
    a.last1[s] = 0;
  }
  return a;
}
// a then b
__device__ __forceinline__ SAgg sagg_combine(const SAgg& a, const SAgg& b) {
  SAgg o;
  o.T = stv_compose(a.T, b.T);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t s2 = stv_apply(a.T, uint32_t(s));
    uint32_t bc = 0, bl = 0;
    uint64_t br = 0, bl1 = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (uint32_t(q) == s2) { bc = b.col[q]; bl = b.lst[q]; br = b.rec[q]; bl1 = b.last1[q]; }
    o.rec[s] = a.rec[s] + br;
    o.col[s] = (bc & ABS32) ? bc : ((a.col[s] & ABS32) | ((a.col[s] + bc) & ~ABS32));
    const bool hb = bl1 != 0;
    o.last1[s] = hb ? bl1 : a.last1[s];
    o.lst[s] = hb ? bl : a.lst[s];
  }
  return o;
}
__device__ __forceinline__ void sagg_pack(const SAgg& a, uint64_t (&w)[13]) {
  w[0] = a.T;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    w[1 + 3 * s] = a.rec[s];
    w[2 + 3 * s] = a.last1[s];
    w[3 + 3 * s] = uint64_t(a.col[s]) | (uint64_t(a.lst[s]) << 32);
  }
}
__device__ __forceinline__ SAgg sagg_unpack(const uint64_t (&w)[13]) {
  SAgg a;
  a.T = uint32_t(w[0]);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    a.rec[s] = w[1 + 3 * s];
    a.last1[s] = w[2 + 3 * s];
    a.col[s] = uint32_t(w[3 + 3 * s]);
    a.lst[s] = uint32_t(w[3 + 3 * s] >> 32);
  }
  return a;
}
__device__ __forceinline__ SAgg sagg_shfl_up(const SAgg& a, int d) {
  uint64_t w[13];
  sagg_pack(a, w);
#pragma unroll
  for (int k = 0; k < 13; ++k) w[k] = __shfl_up_sync(FULL, w[k], d);
  return sagg_unpack(w);
}
struct SAggOp {
  __device__ void operator()(const uint64_t (&a)[13], const uint64_t (&b)[13],
                             uint64_t (&o)[13]) const {
    sagg_pack(sagg_combine(sagg_unpack(a), sagg_unpack(b)), o);
  }
};
__device__ __forceinline__ SAgg sagg_of_tile(const uint8_t* rec, uint64_t tile_base) {
  const uint32_t* h = reinterpret_cast<const uint32_t*>(rec);
  SAgg a;
  a.T = h[0];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    a.rec[s] = h[1 + 3 * s];
    a.col[s] = h[2 + 3 * s];
    const uint32_t l = h[3 + 3 * s];
    a.last1[s] = l ? tile_base + (l >> 8) : 0ull;
    a.lst[s] = l & 0xFFu;
  }
  return a;
}

struct PreHdr {
  uint64_t rec0;     // record index at the tile start
  uint64_t last1;    // global position + 1 of the last terminator before the tile, 0 none
  uint32_t col_in;   // absolute column at the tile start (saturated)
  uint32_t state;    // DFA state at the tile start | state after that terminator << 8
};
constexpr int PRE_HDR = sizeof(PreHdr);

struct ScanShared {
  uint32_t block;
  uint64_t wagg[SCAN_NT / 32][13];
  uint64_t pre[13];
  uint64_t wsum[SCAN_NT / 32][ppi::MAX_STR_COLS];
  uint64_t base[ppi::MAX_STR_COLS];
  int8_t stridx[PP_MAX_COLS];
};

template <int NS>
__global__ void __launch_bounds__(SCAN_NT) scan_kernel(const __grid_constant__ ParseParams P) {
  constexpr int SW = SCAN_NT / 32;
  constexpr int K3 = NS > 0 ? NS : 1;
  __shared__ ScanShared S;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int k = t; k < PP_MAX_COLS; k += SCAN_NT) S.stridx[k] = P.stridx[k];
  if (t == 0) S.block = atomicAdd(&P.s.counters[2], 1u);
  __syncthreads();
  const uint32_t blk = S.block;
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t t0 = blk * SCAN_TILES + uint32_t(t) * SCAN_TPT;
  const uint32_t n_cols = uint32_t(P.n_cols);

  // (A) per-start-state scan of (transition vector, records, column, last terminator)
  SAgg mine = sagg_identity(false);
  for (int i = 0; i < SCAN_TPT; ++i) {
    const uint32_t tile = t0 + i;
    if (tile < P.n_tiles)
      mine = sagg_combine(mine, sagg_of_tile(P.s.ctx + size_t(tile) * P.s.ctx_stride,
                                             uint64_t(tile) * TILE));
  }
  SAgg inc = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const SAgg o = sagg_shfl_up(inc, d);
    if (lane >= d) inc = sagg_combine(o, inc);
  }
  SAgg lex = sagg_shfl_up(inc, 1);
  if (lane == 0) lex = sagg_identity(false);
  if (lane == 31) sagg_pack(inc, S.wagg[warp]);
  __syncthreads();
  if (warp == 0) {
    uint64_t wv[13];
    SAgg x = sagg_identity(false);
    if (lane < SW) {
#pragma unroll
      for (int k = 0; k < 13; ++k) wv[k] = S.wagg[lane][k];
      x = sagg_unpack(wv);
    }
#pragma unroll
    for (int d = 1; d < SW; d <<= 1) {
      const SAgg o = sagg_shfl_up(x, d);
      if (lane >= d) x = sagg_combine(o, x);
    }
    SAgg xe = sagg_shfl_up(x, 1);
    if (lane == 0) xe = sagg_identity(false);
    __syncwarp();
    if (lane < SW) sagg_pack(xe, S.wagg[lane]);
    uint64_t agg[13], seed[13], ident[13], ex[13];
    {
      uint64_t tw[13];
      sagg_pack(x, tw);
#pragma unroll
      for (int k = 0; k < 13; ++k) agg[k] = __shfl_sync(FULL, tw[k], SW - 1);
    }
    sagg_pack(sagg_identity(true), seed);
    sagg_pack(sagg_identity(false), ident);
    lookback_vec<13>(P.s.scan_flag_a, P.s.scan_agg_a, P.s.scan_inc_a, blk, agg, seed, ident,
                     SAggOp{}, cfg, ex);
    if (lane == 0)
#pragma unroll
      for (int k = 0; k < 13; ++k) S.pre[k] = ex[k];
  }
  __syncthreads();
  // resolve this thread's first tile at the true start state
  SAgg blockpre;
  {
    uint64_t pw[13], ww[13];
#pragma unroll
    for (int k = 0; k < 13; ++k) { pw[k] = S.pre[k]; ww[k] = S.wagg[warp][k]; }
    blockpre = sagg_combine(sagg_unpack(pw), sagg_combine(sagg_unpack(ww), lex));
  }
  const uint32_t s0 = P.start_state;
  uint32_t s = stv_apply(blockpre.T, s0);
  uint64_t rec = 0, last1 = 0;
  uint32_t col = 0, lst = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (uint32_t(q) == s0) {
      rec = blockpre.rec[q];
      last1 = blockpre.last1[q];
      col = blockpre.col[q] & ~ABS32;
      lst = blockpre.lst[q];
    }

  // walk this thread's tiles with the true context; per tile, its value
  // bytes per string column follow from its start state and column
  uint64_t sum[K3];
#pragma unroll
  for (int k = 0; k < K3; ++k) sum[k] = 0;
  for (int i = 0; i < SCAN_TPT; ++i) {
    const uint32_t tile = t0 + i;
    if (tile >= P.n_tiles) break;
    const uint8_t* cr = P.s.ctx + size_t(tile) * P.s.ctx_stride;
    uint8_t* pr = P.s.pre + size_t(tile) * P.s.pre_stride;
    PreHdr h;
    h.rec0 = rec;
    h.last1 = last1;
    h.col_in = col;
    h.state = s | (lst << 8);
    *reinterpret_cast<PreHdr*>(pr) = h;
    const uint32_t* hd = reinterpret_cast<const uint32_t*>(cr);
    if (NS > 0) {
      uint64_t* cb = reinterpret_cast<uint64_t*>(pr + PRE_HDR);
      const uint16_t* cabs = reinterpret_cast<const uint16_t*>(cr + CTX_HDR);
      const uint16_t* crel = cabs + 4 * P.n_str;
      uint64_t contrib[K3];
#pragma unroll
      for (int k = 0; k < K3; ++k) contrib[k] = 0;
      if (s < 4) {
#pragma unroll
        for (int k = 0; k < K3; ++k)
          if (k < P.n_str) contrib[k] = cabs[s * P.n_str + k];
        for (uint32_t k = 0; col + k < n_cols; ++k) {
          const int si = S.stridx[col + k];
          const uint32_t v = crel[s * n_cols + k];
          if (si >= 0 && v) {
#pragma unroll
            for (int q = 0; q < K3; ++q)
              if (q == si) contrib[q] += v;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < K3; ++k) {
        if (k < P.n_str) cb[k] = contrib[k];
        sum[k] += contrib[k];
      }
    }
    if (s < 4) {
      const uint32_t trec = hd[1 + 3 * s], tcol = hd[2 + 3 * s], tl = hd[3 + 3 * s];
      rec += trec;
      if (tcol & ABS32) col = tcol & ~ABS32;
      else col = (uint64_t(col) + tcol > 0x7FFFFF00ull) ? 0x7FFFFF00u : col + tcol;
      if (tl) { last1 = uint64_t(tile) * TILE + (tl >> 8); lst = tl & 0xFFu; }
      s = stv_apply(hd[0], s);
    }
  }

  // (C) chars offsets: exclusive sum over tiles per string column
  if (NS > 0) {
    uint64_t ci[K3];
#pragma unroll
    for (int k = 0; k < K3; ++k) ci[k] = sum[k];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
      for (int k = 0; k < K3; ++k) {
        const uint64_t o = __shfl_up_sync(FULL, ci[k], d);
        if (lane >= d) ci[k] += o;
      }
    }
    if (lane == 31)
#pragma unroll
      for (int k = 0; k < K3; ++k) S.wsum[warp][k] = ci[k];
    __syncthreads();
    if (warp == 0) {
      uint64_t v[K3], x[K3], agg[K3], zero[K3], ex[K3];
#pragma unroll
      for (int k = 0; k < K3; ++k) { v[k] = lane < SW ? S.wsum[lane][k] : 0ull; x[k] = v[k]; zero[k] = 0; }
#pragma unroll
      for (int d = 1; d < SW; d <<= 1) {
#pragma unroll
        for (int k = 0; k < K3; ++k) {
          const uint64_t o = __shfl_up_sync(FULL, x[k], d);
          if (lane >= d) x[k] += o;
        }
      }
#pragma unroll
      for (int k = 0; k < K3; ++k) {
        agg[k] = __shfl_sync(FULL, x[k], SW - 1);
        if (lane < SW) S.wsum[lane][k] = x[k] - v[k];
      }
      lookback_vec<K3>(P.s.scan_flag_c, P.s.scan_agg_c, P.s.scan_inc_c, blk, agg, zero, zero,
                       AddOp<K3>{}, cfg, ex);
      if (lane == 0)
#pragma unroll
        for (int k = 0; k < K3; ++k) S.base[k] = ex[k];
    }
    __syncthreads();
    uint64_t run[K3];
#pragma unroll
    for (int k = 0; k < K3; ++k) run[k] = S.base[k] + S.wsum[warp][k] + (ci[k] - sum[k]);
    for (int i = 0; i < SCAN_TPT; ++i) {
      const uint32_t tile = t0 + i;
      if (tile >= P.n_tiles) break;
      uint64_t* cb = reinterpret_cast<uint64_t*>(P.s.pre + size_t(tile) * P.s.pre_stride + PRE_HDR);
#pragma unroll
      for (int k = 0; k < K3; ++k)
        if (k < P.n_str) {
          const uint64_t c = cb[k];
          cb[k] = run[k];
          run[k] += c;
        }
    }
  }
}

// Convert the numeric field in slot value v (tile-relative start << 16 |
// end; start 0xFFFF = the field began in an earlier tile) and store it at
// row `rec` of column c of type ty; reports syntax / range errors.
__device__ __forceinline__ void convert_slot(const ParseParams& P, uint32_t c, uint32_t ty,
                                             uint32_t v, uint64_t rec, uint64_t tile_base,
                                             uint64_t tile_fstart, uint32_t tile_fstate,
                                             const uint8_t* tile_s, const uint32_t* tile_w,
                                             const uint32_t* ctrl_s, const uint32_t* my_lut) {
  uint64_t val = 0;
  int err = 0;
  uint64_t fs = 0;
  if (v != SLOT_DEFAULT) {
    const uint32_t fsr = v >> 16;
    const uint64_t fe = tile_base + (v & 0xFFFFu);
    fs = fsr == 0xFFFFu ? tile_fstart : tile_base + fsr;
    const uint32_t fl = (v & 0xFFFFu) - fsr;
    bool done = false;
    if (fsr != 0xFFFFu && fl > 0 && popc_range(ctrl_s, fsr, fsr + fl) == 0) {
      bool neg;
      if (ty == PP_COL_FLOAT64) {
        uint64_t mant;
        int q;
        if (fast_float(tile_w, fsr, fl, mant, q, neg)) {
          val = (mant ? ppn::decimal_to_binary64(mant, q) : 0ull) | (neg ? (1ull << 63) : 0ull);
          done = true;
        }
      } else {
        uint64_t mag;
        if (fast_int(tile_w, fsr, fl, mag, neg)) {
          const uint64_t lim = ty == PP_COL_INT8 ? (neg ? 128ull : 127ull)
                             : ty == PP_COL_INT32 ? (neg ? 2147483648ull : 2147483647ull)
                             : (neg ? 9223372036854775808ull : 9223372036854775807ull);
          if (mag > lim) err = PP_ERR_NUM_OVERFLOW;
          else val = neg ? (~mag + 1) : mag;
          done = true;
        }
      }
    }
    if (done) {
    } else if (ty == PP_COL_FLOAT64) {
      ppn::FloatAcc acc;
      const uint32_t nd = feed_field(acc, P.in, fs, fe, tile_base, tile_s, ctrl_s, my_lut,
                                     tile_fstate);
      if (nd) err = acc.finish(&val);
    } else {
      ppn::IntAcc acc;
      const uint32_t nd = feed_field(acc, P.in, fs, fe, tile_base, tile_s, ctrl_s, my_lut,
                                     tile_fstate);
      if (nd) {
        int64_t x = 0;
        if (ty == PP_COL_INT8) err = acc.finish(128ull, 127ull, &x);
        else if (ty == PP_COL_INT32) err = acc.finish(2147483648ull, 2147483647ull, &x);
        else err = acc.finish(9223372036854775808ull, 9223372036854775807ull, &x);
        val = uint64_t(x);
      }
    }
  }
  if (ty == PP_COL_FLOAT64) static_cast<uint64_t*>(P.typed[c])[rec] = val;
  else if (ty == PP_COL_INT8) static_cast<int8_t*>(P.typed[c])[rec] = int8_t(val);
  else if (ty == PP_COL_INT32) static_cast<int32_t*>(P.typed[c])[rec] = int32_t(val);
  else static_cast<int64_t*>(P.typed[c])[rec] = int64_t(val);
  if (err) report(P.st, err, fs, true);
}

// ================================================================ 3. main
struct MainShared {
  Feed F;
  uint32_t tile_stv;
  uint32_t rows;             // records touched by the tile (#RD + 1)
  uint32_t warp_stv[NW];
  uint32_t warp_rec[NW], warp_col[NW], warp_last[NW];
  uint64_t wcnt[NW][4];
  uint64_t base[ppi::MAX_STR_COLS];
  uint32_t total[ppi::MAX_STR_COLS];
  uint32_t R[ppi::MAX_STR_COLS];
  int8_t stridx[PP_MAX_COLS];
  uint8_t coltype[PP_MAX_COLS];
  uint8_t outcol[PP_MAX_COLS];  // columns that produce output, in order
  uint8_t numcol[PP_MAX_COLS];  // numeric output columns, in order
  uint32_t n_out, n_num;
  uint32_t wnt[NW];          // per warp: terminators (then exclusive prefix)
  uint32_t nterm;            // terminators in the tile
  uint32_t wrd[NW], crd[NW]; // per warp range: record delimiters, carry in
  int32_t wlast[NW], clast[NW], lastrd;
  uint32_t cstart[ppi::MAX_STR_COLS + 1];
};
constexpr int LIST_CAP = 4096;         // terminators per tile on the field-list path
constexpr size_t MAIN_SMEM = LUT_BYTES + 2 * TILE + STAGE_BYTES + SLOT_CAP * 4 + NT * 4 +
                             LIST_CAP * 2 + sizeof(MainShared);

template <int NS>
__global__ void __launch_bounds__(NT, 2) main_kernel(const __grid_constant__ ParseParams P) {
  constexpr int NSW = NS > 0 ? (NS + 3) / 4 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin0 = smem + LUT_BYTES;             // two tile buffers
  uint8_t* stage_s = lin0 + 2 * TILE;
  uint32_t* slot_s = reinterpret_cast<uint32_t*>(stage_s + STAGE_BYTES);
  uint32_t* ctrl_s = slot_s + SLOT_CAP;
  uint16_t* list_s = reinterpret_cast<uint16_t*>(ctrl_s + NT);  // field list, then chars ends
  MainShared& S = *reinterpret_cast<MainShared*>(list_s + LIST_CAP);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  load_lut(P, lut_s);
  for (int k = t; k < PP_MAX_COLS; k += NT) {
    S.stridx[k] = P.stridx[k];
    S.coltype[k] = P.coltype[k];
  }
  if (t == 0) {
    uint32_t k = 0, m = 0;
    for (uint32_t c = 0; c < uint32_t(P.n_cols); ++c) {
      if (P.coltype[c] != PP_COL_SKIP) S.outcol[k++] = uint8_t(c);
      if (P.coltype[c] != PP_COL_SKIP && P.coltype[c] != PP_COL_STRING) S.numcol[m++] = uint8_t(c);
    }
    S.n_out = k;
    S.n_num = m;
  }
  const uint32_t* my_lut = lut_s + lane;
  const uint32_t n_cols = uint32_t(P.n_cols);
  const bool aligned_in = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;
  uint32_t* counter = &P.s.counters[1];
  feed_start(P, S.F, counter, aligned_in, lin0);

  for (;;) {
    const uint32_t tile = S.F.tile[S.F.cur];
    if (tile >= P.n_tiles) break;
    uint8_t* tile_s = lin0 + S.F.cur * TILE;
    const uint32_t* tile_w = reinterpret_cast<const uint32_t*>(tile_s);
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    const bool last_tile = tile + 1 == P.n_tiles;
    const uint8_t* pr = P.s.pre + size_t(tile) * P.s.pre_stride;
    const PreHdr ph = *reinterpret_cast<const PreHdr*>(pr);
    uint32_t w[8];
    feed_tile(P, S.F, tile_s, tile_base, tile_len, w);
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    const uint8_t* own = tile_s + cstart;

    // ---- context resolution: the tile's start state is known from the scan
    uint32_t G, special, special_x;
    stv_pass(w, clen, tile_s, cstart, my_lut, G, special, special_x);
    const uint32_t lane_ex = block_stv(G, S.warp_stv, &S.tile_stv);
    const uint32_t s_tile = ph.state & 0xFFu;
    const uint32_t s_chunk = stv_apply(lane_ex, stv_apply(S.warp_stv[warp], s_tile));

    // ---- tagging
    const Tags g = tag_chunk(s_chunk, special, special_x, P.sticky, clen, cstart, own, my_lut,
                             P.bg_next);
    const uint32_t fd = g.fd, rd = g.rd;
    const uint32_t valid = range_mask(0, min(clen, g.inv_at));
    const uint32_t data = valid & ~(fd | rd | g.ctrl);
    ctrl_s[t] = g.ctrl;
    if (g.inv_at < clen && s_chunk != 4)
      report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + g.inv_at, true);
    const bool owns_end = last_tile && clen > 0 && cstart + clen == tile_len;
    if (owns_end && g.end != 4 && !((P.accept_mask >> g.end) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    const bool virt_rd = owns_end && g.end != 4 && ((P.accept_mask >> g.end) & 1u) &&
                         !((rd >> (clen - 1)) & 1u);

    // ---- record and column indices across the block (tile prefix from the scan)
    V2 vi = chunk_v2(g);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const V2 o = shfl_up_v2(vi, d);
      if (lane >= d) vi = op2_32(o, vi);
    }
    V2 lex = shfl_up_v2(vi, 1);
    if (lane == 0) lex = {0u, 0u, 0u};
    if (lane == 31) { S.warp_rec[warp] = vi.rec; S.warp_col[warp] = vi.col; S.warp_last[warp] = vi.last; }
    __syncthreads();
    if (warp == 0) {
      V2 x = lane < NW ? V2{S.warp_rec[lane], S.warp_col[lane], S.warp_last[lane]} : V2{0u, 0u, 0u};
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const V2 o = shfl_up_v2(x, d);
        if (lane >= d) x = op2_32(o, x);
      }
      V2 xe = shfl_up_v2(x, 1);
      if (lane == 0) xe = {0u, 0u, 0u};
      __syncwarp();
      if (lane < NW) { S.warp_rec[lane] = xe.rec; S.warp_col[lane] = xe.col; S.warp_last[lane] = xe.last; }
      if (lane == NW - 1) S.rows = x.rec + 1;
    }
    __syncthreads();
    const V2 pre = op2_32(V2{S.warp_rec[warp], S.warp_col[warp], S.warp_last[warp]}, lex);
    const uint64_t tile_rec0 = ph.rec0;
    const uint64_t rec0 = tile_rec0 + pre.rec;
    uint32_t col0;
    if (pre.col & ABS32) {
      col0 = pre.col & ~ABS32;
    } else {
      const uint64_t c = uint64_t(ph.col_in) + pre.col;
      col0 = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
    }
    const uint64_t fstart0 = pre.last ? tile_base + (pre.last >> 8) : ph.last1;
    // start (global) and DFA state of the field holding tile byte 0
    const uint64_t tile_fstart = ph.last1;
    const uint32_t tile_fstate = ph.last1 ? (ph.state >> 8) & 0xFFu : uint32_t(P.start_state);

    // ---- terminators of the tile (field ends): count and block scan
    const uint32_t term_mask = fd | rd;
    {
      const uint32_t nt = __popc(term_mask) + (virt_rd ? 1u : 0u);
      uint32_t ti = nt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, ti, d);
        if (lane >= d) ti += o;
      }
      if (lane == 31) S.wnt[warp] = ti;
      __syncthreads();
      if (warp == 0) {
        const uint32_t v = lane < NW ? S.wnt[lane] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int d = 1; d < NW; d <<= 1) {
          const uint32_t o = __shfl_up_sync(FULL, x, d);
          if (lane >= d) x += o;
        }
        __syncwarp();
        if (lane < NW) S.wnt[lane] = x - v;
        if (lane == NW - 1) S.nterm = x;
      }
      __syncthreads();
      if (S.nterm <= LIST_CAP && n_cols * S.rows <= SLOT_CAP) {
        uint32_t i = S.wnt[warp] + ti - nt;
        uint32_t m = term_mask;
        while (m) {
          const uint32_t j = __ffs(m) - 1;
          m &= m - 1;
          list_s[i++] = uint16_t((cstart + j) | (((rd >> j) & 1u) << 15));
        }
        if (virt_rd) list_s[i] = uint16_t(tile_len | 0x8000u);
      }
      __syncthreads();  // the list is read across warps below
    }
    const uint32_t T = S.nterm;
    const uint32_t rows = S.rows;
    uint64_t rec_end = rec0;
    if (T <= LIST_CAP && n_cols * rows <= SLOT_CAP) {
      // ======== field-list path: one lane per field, warp ranges with carries
      for (uint32_t k = t; k < n_cols * rows; k += NT) slot_s[k] = SLOT_ABSENT;
      const uint32_t R = (((T + NW - 1) / NW) + 31u) & ~31u;
      const uint32_t r0 = min(T, uint32_t(warp) * R), r1 = min(T, r0 + R);
      {
        uint32_t nrd = 0;
        int32_t last = -1;
        for (uint32_t g0 = r0; g0 < r1; g0 += 32) {
          const uint32_t f = g0 + lane;
          const uint32_t b = __ballot_sync(FULL, f < r1 && (list_s[f] >> 15));
          nrd += __popc(b);
          if (b) last = int32_t(g0 + 31 - __clz(b));
        }
        if (lane == 0) { S.wrd[warp] = nrd; S.wlast[warp] = last; }
      }
      __syncthreads();
      if (t == 0) {
        uint32_t cnt = 0;
        int32_t lst = -1;
        for (int q = 0; q < NW; ++q) {
          S.crd[q] = cnt;
          S.clast[q] = lst;
          cnt += S.wrd[q];
          if (S.wlast[q] >= 0) lst = S.wlast[q];
        }
        S.lastrd = lst;
      }
      __syncthreads();
      const uint32_t first_in = tile_fstart >= tile_base ? 0u : 0xFFFFu;  // start of field 0
      {
        uint32_t crd = S.crd[warp];
        int32_t clast = S.clast[warp];
        const uint32_t lt = (1u << lane) - 1u;
        for (uint32_t g0 = r0; g0 < r1; g0 += 32) {
          const uint32_t f = g0 + lane;
          const bool ok = f < r1;
          const uint32_t e = ok ? uint32_t(list_s[f]) : 0u;
          const bool isrd = ok && (e >> 15);
          const uint32_t b = __ballot_sync(FULL, isrd);
          if (ok) {
            const uint32_t below = b & lt;
            const uint32_t rl = crd + __popc(below);
            const int32_t lr = below ? int32_t(g0 + 31 - __clz(below)) : clast;
            uint32_t col;
            if (lr >= 0) {
              col = f - uint32_t(lr) - 1u;
            } else {
              const uint64_t cc = uint64_t(ph.col_in) + f;
              col = cc > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(cc);
            }
            const uint32_t pos = e & 0x7FFFu;
            const uint32_t s0 = f ? (uint32_t(list_s[f - 1]) & 0x7FFFu) + 1u : first_in;
            if (col < n_cols && S.coltype[col] != PP_COL_SKIP) slot_s[col * rows + rl] = (s0 << 16) | pos;
            if (isrd && col != n_cols - 1) {
              report(P.st, PP_ERR_COLCOUNT, tile_base + pos, true);
              for (uint32_t c = col + 1; c < n_cols; ++c)
                if (S.coltype[c] != PP_COL_SKIP) slot_s[c * rows + rl] = SLOT_DEFAULT;
            }
          }
          crd += __popc(b);
          if (b) clast = int32_t(g0 + 31 - __clz(b));
        }
      }
      if (NS > 0 && t == 0) {  // the field still open at the tile end: value bytes only
        const uint32_t s0 = T ? (uint32_t(list_s[T - 1]) & 0x7FFFu) + 1u : first_in;
        const uint32_t s0in = s0 == 0xFFFFu ? 0u : s0;
        if (s0in < tile_len) {
          uint32_t col;
          if (S.lastrd >= 0) {
            col = T - uint32_t(S.lastrd) - 1u;
          } else {
            const uint64_t cc = uint64_t(ph.col_in) + T;
            col = cc > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(cc);
          }
          if (col < n_cols && S.stridx[col] >= 0)
            slot_s[col * rows + rows - 1] = (s0 << 16) | tile_len | 0x8000u;
        }
      }
      __syncthreads();
      // string columns: value bytes per field -> chars end offsets (a block
      // scan over the column-major string slots), tile totals, staging layout
      const uint32_t n_str = uint32_t(P.n_str);
      if (NS > 0 && n_str) {
        const uint32_t n = n_str * rows;
        const uint32_t per = (n + NT - 1) / NT;
        const uint32_t k0 = min(n, uint32_t(t) * per), k1 = min(n, k0 + per);
        uint32_t lens[8];
        uint32_t mysum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t k = k0 + q;
          uint32_t len = 0;
          if (k < k1) {
            const uint32_t si = k / rows, r = k - si * rows;
            const uint32_t v = slot_s[P.strcol[si] * rows + r];
            if (v != SLOT_ABSENT && v != SLOT_DEFAULT) {
              const uint32_t a0 = (v >> 16) == 0xFFFFu ? 0u : (v >> 16), e = v & 0x7FFFu;
              len = (e - a0) - popc_range(ctrl_s, a0, e);
            }
          }
          lens[q] = len;
          mysum += len;
        }
        uint32_t xi = mysum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(FULL, xi, d);
          if (lane >= d) xi += o;
        }
        if (lane == 31) S.wnt[warp] = xi;
        __syncthreads();
        if (warp == 0) {
          const uint32_t v = lane < NW ? S.wnt[lane] : 0u;
          uint32_t x = v;
#pragma unroll
          for (int d = 1; d < NW; d <<= 1) {
            const uint32_t o = __shfl_up_sync(FULL, x, d);
            if (lane >= d) x += o;
          }
          __syncwarp();
          if (lane < NW) S.wnt[lane] = x - v;
          if (lane == NW - 1) S.cstart[n_str] = x;
        }
        __syncthreads();
        uint32_t run = S.wnt[warp] + xi - mysum;  // exclusive prefix of item k0
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t k = k0 + q;
          if (k < k1) {
            if (k % rows == 0) S.cstart[k / rows] = run;
            run += lens[q];
            list_s[k] = uint16_t(run);  // inclusive: end of the field's chars in the tile
          }
        }
        __syncthreads();
        for (uint32_t k = t; k < n; k += NT) list_s[k] = uint16_t(list_s[k] - S.cstart[k / rows]);
        if (t == 0) {
          const uint64_t* cb = reinterpret_cast<const uint64_t*>(pr + PRE_HDR);
          uint32_t Rr = 0;
          for (uint32_t c = 0; c < n_str; ++c) {
            const uint32_t a = S.cstart[c + 1] - S.cstart[c];
            const uint64_t b = cb[c];
            S.base[c] = b;
            S.total[c] = a;
            const uintptr_t gp = reinterpret_cast<uintptr_t>(P.chars[c]) + b;
            Rr = ((Rr + 15u) & ~15u) + uint32_t(gp & 15u);
            S.R[c] = Rr;
            Rr += a;
            if (last_tile) P.st->chars_len[P.strcol[c]] = b + a;
          }
        }
        __syncthreads();
        // Arrow offsets of closed string fields (coalesced per column)
        for (uint32_t k = t; k < n; k += NT) {
          const uint32_t si = k / rows, r = k - si * rows;
          const uint32_t v = slot_s[P.strcol[si] * rows + r];
          if (v == SLOT_ABSENT || (v != SLOT_DEFAULT && (v & 0x8000u))) continue;
          const uint64_t rec = tile_rec0 + r;
          if (!P.has_out) continue;
          if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
          const uint64_t off = S.base[si] + list_s[k];
          if (off > 0x7FFFFFFFull || off > P.chars_cap[si]) report(P.st, PP_ERR_CAPACITY, 0, false);
          else P.offsets[si][rec + 1] = int32_t(off);
        }
        // stage value bytes: a lane per short field, a warp per long one
        for (uint32_t k = t; k < n; k += NT) {
          const uint32_t si = k / rows, r = k - si * rows;
          const uint32_t v = slot_s[P.strcol[si] * rows + r];
          if (v == SLOT_ABSENT || v == SLOT_DEFAULT) continue;
          const uint32_t a0 = (v >> 16) == 0xFFFFu ? 0u : (v >> 16), e = v & 0x7FFFu;
          if (e - a0 > 64 || popc_range(ctrl_s, a0, e)) continue;
          uint32_t dst = S.R[si] + list_s[k] - (e - a0);
          for (uint32_t p = a0; p < e; ++p) stage_s[dst++] = uint8_t(tile_byte(tile_s, p));
        }
        for (uint32_t k = warp; k < n; k += NW) {
          const uint32_t si = k / rows, r = k - si * rows;
          const uint32_t v = slot_s[P.strcol[si] * rows + r];
          if (v == SLOT_ABSENT || v == SLOT_DEFAULT) continue;
          const uint32_t a0 = (v >> 16) == 0xFFFFu ? 0u : (v >> 16), e = v & 0x7FFFu;
          const uint32_t nctrl = popc_range(ctrl_s, a0, e);
          if (e - a0 <= 64 && !nctrl) continue;
          const uint32_t len = (e - a0) - nctrl;
          uint32_t dst = S.R[si] + list_s[k] - len;
          for (uint32_t p0 = a0; p0 < e; p0 += 32) {
            const uint32_t p = p0 + lane;
            const bool isdata = p < e && !((ctrl_s[p >> 5] >> (p & 31)) & 1u);
            const uint32_t bb = __ballot_sync(FULL, isdata);
            if (isdata) stage_s[dst + __popc(bb & ((1u << lane) - 1u))] = uint8_t(tile_byte(tile_s, p));
            dst += __popc(bb);
          }
        }
      }
      // numbers: a warp per 32 rows of one column
      if (P.has_out && S.n_num) {
        const uint32_t nch = (rows + 31) / 32;
        const uint32_t total = S.n_num * nch;
        for (uint32_t ci = warp; ci < total; ci += NW) {
          const uint32_t oc = ci / nch;
          const uint32_t r = (ci - oc * nch) * 32 + lane;
          const uint32_t c = S.numcol[oc];
          if (r >= rows) continue;
          const uint32_t v = slot_s[c * rows + r];
          if (v == SLOT_ABSENT) continue;
          const uint64_t rec = tile_rec0 + r;
          if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
          convert_slot(P, c, S.coltype[c], v, rec, tile_base, tile_fstart, tile_fstate, tile_s,
                       tile_w, ctrl_s, my_lut);
        }
      }
      __syncthreads();
      rec_end = tile_rec0 + (rows - 1) + (virt_rd ? 1u : 0u);
    } else {
      // ======== general path: per-thread walk over the chunk's fields
      // ---- value bytes per string column: block scan, staging layout
      uint64_t cex[NSW];
  #pragma unroll
      for (int k = 0; k < NSW; ++k) cex[k] = 0;
      if (NS > 0) {
        uint64_t cnt[NSW];
  #pragma unroll
        for (int k = 0; k < NSW; ++k) cnt[k] = 0;
        {
          uint32_t term = fd | rd, col = col0, start = 0;
          for (;;) {
            const uint32_t j = term ? uint32_t(__ffs(term) - 1) : 32u;
            const uint32_t seg = data & range_mask(start, j);
            if (col < n_cols) {
              const int si = S.stridx[col];
              if (si >= 0) add16(cnt, si, __popc(seg));
            }
            if (j == 32) break;
            col = ((rd >> j) & 1u) ? 0u : col + 1;
            start = j + 1;
            term &= term - 1;
          }
        }
        uint64_t ci[NSW];
  #pragma unroll
        for (int k = 0; k < NSW; ++k) ci[k] = cnt[k];
  #pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
  #pragma unroll
          for (int k = 0; k < NSW; ++k) {
            const uint64_t o = __shfl_up_sync(FULL, ci[k], d);
            if (lane >= d) ci[k] += o;
          }
        }
        if (lane == 31) {
  #pragma unroll
          for (int k = 0; k < NSW; ++k) S.wcnt[warp][k] = ci[k];
        }
        __syncthreads();
        if (warp == 0) {
          uint64_t wv[NSW], wi2[NSW];
  #pragma unroll
          for (int k = 0; k < NSW; ++k) { wv[k] = lane < NW ? S.wcnt[lane][k] : 0ull; wi2[k] = wv[k]; }
  #pragma unroll
          for (int d = 1; d < NW; d <<= 1) {
  #pragma unroll
            for (int k = 0; k < NSW; ++k) {
              const uint64_t o = __shfl_up_sync(FULL, wi2[k], d);
              if (lane >= d) wi2[k] += o;
            }
          }
          uint64_t tot[NSW];
  #pragma unroll
          for (int k = 0; k < NSW; ++k) {
            tot[k] = __shfl_sync(FULL, wi2[k], NW - 1);
            if (lane < NW) S.wcnt[lane][k] = wi2[k] - wv[k];
          }
          if (lane == 0) {
            const uint64_t* cb = reinterpret_cast<const uint64_t*>(pr + PRE_HDR);
            uint32_t R = 0;
  #pragma unroll
            for (int c = 0; c < NS; ++c) {
              if (c < P.n_str) {
                const uint32_t a = uint32_t((tot[c >> 2] >> (16 * (c & 3))) & 0xFFFFull);
                const uint64_t b = cb[c];
                S.base[c] = b;
                S.total[c] = a;
                const uintptr_t gp = reinterpret_cast<uintptr_t>(P.chars[c]) + b;
                R = ((R + 15u) & ~15u) + uint32_t(gp & 15u);
                S.R[c] = R;
                R += a;
                if (last_tile) P.st->chars_len[P.strcol[c]] = b + a;
              }
            }
          }
        }
        __syncthreads();
  #pragma unroll
        for (int k = 0; k < NSW; ++k) cex[k] = S.wcnt[warp][k] + (ci[k] - cnt[k]);
      }

      // ---- fields: staging + (column, record) slots, then one lane per field
      const uint32_t rows = S.rows;
      const uint32_t n_out = S.n_out;
      const uint32_t rpb = max(1u, uint32_t(SLOT_CAP) / n_cols);  // rows per pass
      for (uint32_t lo = 0; lo < rows; lo += rpb) {
        const uint32_t hi = min(rows, lo + rpb);
        const uint32_t nr = hi - lo;
        for (uint32_t k = t; k < n_cols * nr; k += NT) slot_s[k] = SLOT_ABSENT;
        __syncthreads();
        {
          uint32_t term = fd | rd, col = col0, start = 0;
          uint64_t rec = rec0, fstart = fstart0;
          uint64_t loc[NSW];
  #pragma unroll
          for (int k = 0; k < NSW; ++k) loc[k] = 0;
          for (;;) {
            const uint32_t j = term ? uint32_t(__ffs(term) - 1) : 32u;
            const uint32_t seg = data & range_mask(start, j);
            const int si = (NS > 0 && col < n_cols) ? int(S.stridx[col]) : -1;
            if (si >= 0 && seg) {
              if (lo == 0)  // stage this chunk's value bytes once
                stage_runs(seg, S.R[si] + get16(cex, si) + get16(loc, si), own, stage_s);
              add16(loc, si, __popc(seg));
            }
            uint64_t tpos;
            bool is_rd;
            if (j < 32) { tpos = tile_base + cstart + j; is_rd = (rd >> j) & 1u; }
            else if (virt_rd) { tpos = P.n; is_rd = true; }
            else break;
            const uint64_t rl = rec - tile_rec0;
            const bool in_pass = rl >= lo && rl < hi;
            if (in_pass && col < n_cols && S.coltype[col] != PP_COL_SKIP) {
              uint32_t v;
              if (si >= 0) {
                v = get16(cex, si) + get16(loc, si);
              } else {
                const uint32_t fs = fstart >= tile_base ? uint32_t(fstart - tile_base) : 0xFFFFu;
                v = (fs << 16) | uint32_t(tpos - tile_base);
              }
              slot_s[col * nr + uint32_t(rl - lo)] = v;
            }
            if (is_rd) {
              if (col != n_cols - 1) {
                if (lo == 0) report(P.st, PP_ERR_COLCOUNT, tpos, true);
                if (in_pass) {  // missing fields take the column default
                  for (uint32_t c = col + 1; c < n_cols; ++c) {
                    const int sc = S.stridx[c];
                    slot_s[c * nr + uint32_t(rl - lo)] =
                        sc >= 0 ? get16(cex, sc) + get16(loc, sc) : SLOT_DEFAULT;
                  }
                }
              }
              ++rec;
              col = 0;
            } else {
              col = col < 0x7FFFFF00u ? col + 1 : col;
            }
            fstart = tpos + 1;
            if (j == 32) break;
            start = j + 1;
            term &= term - 1;
          }
          rec_end = rec;
        }
        __syncthreads();
        if (P.has_out) {
          const uint32_t items = n_out * nr;
          for (uint32_t k = t; k < items; k += NT) {
            const uint32_t oi = k / nr, r = k - oi * nr;
            const uint32_t c = S.outcol[oi];
            const uint32_t v = slot_s[c * nr + r];
            if (v == SLOT_ABSENT) continue;
            const uint64_t rec = tile_rec0 + lo + r;
            if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
            const uint32_t ty = S.coltype[c];
            if (ty == PP_COL_STRING) {
              const int si = S.stridx[c];
              const uint64_t off = S.base[si] + v;
              if (off > 0x7FFFFFFFull || off > P.chars_cap[si]) report(P.st, PP_ERR_CAPACITY, 0, false);
              else P.offsets[si][rec + 1] = int32_t(off);
              continue;
            }
            convert_slot(P, c, ty, v, rec, tile_base, tile_fstart, tile_fstate, tile_s, tile_w, ctrl_s,
                         my_lut);
          }
        }
        __syncthreads();
      }
    }
    if (owns_end) P.st->n_records = rec_end;

    // ---- staged chars -> HBM
    if (NS > 0 && P.has_out) {
      for (int c = 0; c < P.n_str; ++c) {
        uint32_t len = S.total[c];
        if (!len) continue;
        const uint64_t gb = S.base[c];
        if (gb + len > P.chars_cap[c]) {
          if (t == 0) report(P.st, PP_ERR_CAPACITY, 0, false);
          len = gb >= P.chars_cap[c] ? 0u : uint32_t(P.chars_cap[c] - gb);
        }
        uint8_t* gp = P.chars[c] + gb;
        const uint8_t* sp = stage_s + S.R[c];
        const uint32_t head = min(len, uint32_t((16u - (reinterpret_cast<uintptr_t>(gp) & 15u)) & 15u));
        const uint32_t nvec = (len - head) >> 4;
        const uint32_t tail0 = head + (nvec << 4);
        if (uint32_t(t) < head) gp[t] = sp[t];
        uint4* gv = reinterpret_cast<uint4*>(gp + head);
        const uint4* sv = reinterpret_cast<const uint4*>(sp + head);
        for (uint32_t v = t; v < nvec; v += NT) __stcs(gv + v, sv[v]);
        if (tail0 + t < len) gp[tail0 + t] = sp[tail0 + t];
      }
    }
    feed_next(P, S.F, counter, aligned_in, lin0);  // the tile was last read before a barrier above
  }
  feed_finish(S.F);
}

// ================================================================= launch
// Zero the tile counters and the scan's look-back flags; initialise the
// status and offsets[c][0] = 0 for every string column.
__global__ void parse_init_kernel(uint32_t* counters, uint32_t* flag_a, uint32_t* flag_c,
                                  uint32_t n_blocks, pp_status* st, ParseParams P) {
  const uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x;
  for (uint32_t i = i0; i < n_blocks; i += gridDim.x * blockDim.x) { flag_a[i] = 0; flag_c[i] = 0; }
  if (i0 < 4) counters[i0] = 0;
  if (i0 == 0) {
    st->error = 0;
    st->reserved = 0;
    st->first_error_offset = ~0ull;
    st->n_records = 0;
    st->n_tokens = 0;
    for (int c = 0; c < PP_MAX_COLS; ++c) st->chars_len[c] = 0;
    if (P.has_out)
      for (int c = 0; c < P.n_str; ++c) P.offsets[c][0] = 0;
  }
}

struct Occ { int ctx = -1, main = -1, n_sm = 0; };

template <int NS>
cudaError_t launch_ns(const ParseParams& p, cudaStream_t stream) {
  static Occ occ;
  cudaError_t e;
  if (occ.ctx < 0) {
    int dev;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&occ.n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(ctx_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(CTX_SMEM))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(main_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(MAIN_SMEM))) != cudaSuccess)
      return e;
    int b = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, ctx_kernel<NS>, NT, CTX_SMEM)) !=
        cudaSuccess)
      return e;
    occ.ctx = b > 0 ? b : 1;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, main_kernel<NS>, NT, MAIN_SMEM)) !=
        cudaSuccess)
      return e;
    occ.main = b > 0 ? b : 1;
  }
  const ppi::ParseScratch& s = p.s;
  parse_init_kernel<<<std::max<uint32_t>(1, (s.n_scan_blocks + 255) / 256), 256, 0, stream>>>(
      s.counters, s.scan_flag_a, s.scan_flag_c, s.n_scan_blocks, p.st, p);
  if ((e = cudaGetLastError()) != cudaSuccess || p.n_tiles == 0) return e;
  const uint32_t g1 = uint32_t(std::min<uint64_t>(p.n_tiles, uint64_t(occ.n_sm) * occ.ctx));
  ctx_kernel<NS><<<g1, NT, CTX_SMEM, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  scan_kernel<NS><<<s.n_scan_blocks, SCAN_NT, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const uint32_t g3 = uint32_t(std::min<uint64_t>(p.n_tiles, uint64_t(occ.n_sm) * occ.main));
  main_kernel<NS><<<g3, NT, MAIN_SMEM, stream>>>(p);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
uint32_t ctx_stride_of(int n_str, int n_cols) {
  const size_t b = CTX_HDR + (n_str > 0 ? 8 * size_t(n_str) + 8 * size_t(n_cols) : 0);
  return uint32_t((b + 15) & ~size_t(15));
}
uint32_t pre_stride_of(int n_str) { return uint32_t(PRE_HDR + 8 * (n_str > 0 ? n_str : 0)); }

}  // namespace

namespace ppi {

size_t parse_tile_bytes() { return TILE; }

int parse_ns_width(int n_str) {
  if (n_str <= 0) return 0;
  if (n_str <= 4) return 4;
  if (n_str <= 8) return 8;
  return 16;
}

// layout: counters (16 B) | scan flags a, c | scan payloads a (2 x 13 words
// per block), c (2 x ns words per block) | ctx records | pre records
size_t parse_scratch_bytes(uint32_t n, int ns, int n_cols) {
  const uint32_t nb = (n + SCAN_TILES - 1) / SCAN_TILES;
  const int k3 = ns > 0 ? ns : 1;
  return 256 + 2 * align256(size_t(nb) * 4) + 2 * align256(size_t(nb) * 13 * 8) +
         2 * align256(size_t(nb) * k3 * 8) + align256(size_t(n) * ctx_stride_of(ns, n_cols)) +
         align256(size_t(n) * pre_stride_of(ns));
}

void parse_scratch_carve(void* base, uint32_t n, int ns, int n_cols, ParseScratch* o) {
  const uint32_t nb = (n + SCAN_TILES - 1) / SCAN_TILES;
  const int k3 = ns > 0 ? ns : 1;
  uint8_t* p = static_cast<uint8_t*>(base);
  o->counters = reinterpret_cast<uint32_t*>(p); p += 256;
  o->scan_flag_a = reinterpret_cast<uint32_t*>(p); p += align256(size_t(nb) * 4);
  o->scan_flag_c = reinterpret_cast<uint32_t*>(p); p += align256(size_t(nb) * 4);
  o->scan_agg_a = reinterpret_cast<uint64_t*>(p); p += align256(size_t(nb) * 13 * 8);
  o->scan_inc_a = reinterpret_cast<uint64_t*>(p); p += align256(size_t(nb) * 13 * 8);
  o->scan_agg_c = reinterpret_cast<uint64_t*>(p); p += align256(size_t(nb) * k3 * 8);
  o->scan_inc_c = reinterpret_cast<uint64_t*>(p); p += align256(size_t(nb) * k3 * 8);
  o->ctx = p; p += align256(size_t(n) * ctx_stride_of(ns, n_cols));
  o->pre = p;
  o->ctx_stride = ctx_stride_of(ns, n_cols);
  o->pre_stride = pre_stride_of(ns);
  o->n_scan_blocks = nb;
}

cudaError_t launch_parse(const ParseParams& p, cudaStream_t stream) {
  switch (parse_ns_width(p.n_str)) {
    case 0: return launch_ns<0>(p, stream);
    case 4: return launch_ns<4>(p, stream);
    case 8: return launch_ns<8>(p, stream);
    default: return launch_ns<16>(p, stream);
  }
}

}  // namespace ppi
