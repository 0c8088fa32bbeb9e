// pp_parse: DFA-based parsing of delimiter-separated input into Arrow-style
// columns on sm_103a, in five kernels with no inter-tile waiting on the
// byte-level hot path.
//
// The input is cut into 16 KiB tiles.  In the two tile passes a tile is one
// CTA of 512 threads and each thread owns a 32-byte chunk (one bit per byte
// in the bitmap indexes).  Tiles reach shared memory by a 1-D bulk copy
// (TMA engine) into one of two linear buffers, the next tile's copy running
// while the current one is processed.
//
// 0. Tile start states (tile_stv_kernel, tile_state_kernel).  A warp per
//    tile folds the tile's transition vector (ParPaRaw Section 3.1, Figure
//    2): the vector of the four live states sits in one register, one byte
//    per state, and each byte composes it with its symbol group's row by
//    one byte-permute (the row-per-group transition table of ParPaRaw
//    Section 5, Table 1, read from a per-lane replicated shared-memory LUT).
//    An exclusive composite scan over tiles gives every tile's true start
//    state.
// 1. Context pass (ctx_kernel).  Each thread folds its chunk's vector the
//    same way; vectors compose across the warp (shuffles) and the block,
//    which with the tile's start state gives every chunk's start state.
//    The thread then tags its chunk (one DFA over the non-background bytes
//    only) and the tile records, for its true start state: record count,
//    absolute or relative column offset (ParPaRaw Section 3.2, Figure 4),
//    last terminator, value bytes per string column for fields whose column
//    is known inside the tile, and value bytes per relative field of the
//    tile's first, partial record.  With room in the scratch it also stores
//    every chunk's tag bitmaps and its (record, column, last terminator)
//    prefix inside the tile for the main pass.
// 2. Scan (scan_kernel).  An exclusive scan over tiles with the record-count
//    / column-offset operators (Section 3.2) resolves every tile's record
//    index, column and last terminator; the tile's value bytes per string
//    column then follow from its column, and a second scan turns them into
//    chars offsets.  Blocks chain by a single-pass decoupled look-back.
// 3. Main pass (main_kernel).  With its context known, each tile loads its
//    chunks' tags and prefixes (or, without them, tags again and scans the
//    block), enters every closed field in a column-major (column, record)
//    slot table, compacts string value bytes per column into shared memory
//    (stream compaction in place of ParPaRaw's radix partitioning, Section
//    3.3) and writes them as 16-byte stores; one lane per field then writes
//    the Arrow offset or converts the number (Section 3.3), 32 consecutive
//    rows of a column to a warp for coalesced stores.
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
constexpr uint32_t SLOT_DEFAULT = 0xFFFFFFFDu; // missing field: column default
constexpr uint32_t WAIT_LIMIT = 1u << 24;      // bounded mbarrier polls
constexpr int SCAN_NT = 256;           // scan kernel threads
constexpr int SCAN_TPT = 8;            // tiles per scan thread
constexpr int SCAN_TILES = SCAN_NT * SCAN_TPT;

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

// control bytes before tile position p (p <= tile length)
__device__ __forceinline__ uint32_t ctrl_before(const uint32_t* ctrl_s, const uint16_t* cpre,
                                                uint32_t p) {
  const uint32_t w = p >> 5, b = p & 31u;
  return cpre[w] + (b ? uint32_t(__popc(ctrl_s[w] & ((1u << b) - 1u))) : 0u);
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

__device__ __forceinline__ void load_lut(const ParseParams& P, uint32_t* lut_s) {
  for (int k = threadIdx.x; k < 256 * 32; k += NT) lut_s[k] = P.lut[k >> 5];
}

// ======================================================= 0. tile start states
// The context pass works from each tile's true start state, found first by a
// transition-vector pass (ParPaRaw Section 3.1) and an exclusive composite
// scan over tiles.
constexpr int TV_NT = 256;              // tile-vector pass: a warp per tile
constexpr int TV_BYTES = TILE / 32;     // bytes per lane
constexpr int TS_NT = 256, TS_TPT = 16; // tile-state scan: tiles per thread
constexpr int TS_TILES = TS_NT * TS_TPT;

// Transition vector of each tile: one warp per tile, each lane folding
// TV_BYTES bytes back to front, a warp scan composing the lanes in order.
__global__ void __launch_bounds__(TV_NT) tile_stv_kernel(const __grid_constant__ ParseParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  for (int k = threadIdx.x; k < 256 * 32; k += TV_NT) lut_s[k] = P.lut[k >> 5];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint32_t* my_lut = lut_s + lane;
  const bool aligned = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;
  const uint32_t warps = gridDim.x * (TV_NT / 32);
  for (uint32_t tile = blockIdx.x * (TV_NT / 32) + (threadIdx.x >> 5); tile < P.n_tiles;
       tile += warps) {
    const uint64_t b0 = uint64_t(tile) * TILE + uint64_t(lane) * TV_BYTES;
    const uint32_t len = b0 < P.n ? uint32_t(min(uint64_t(TV_BYTES), P.n - b0)) : 0u;
    uint32_t G = STV_ID;
    if (len == TV_BYTES && aligned) {
      // back to front in steps of 64 bytes, the next step's loads in flight
      // while the current one folds
      constexpr int STEPS = TV_BYTES / 64;
      const uint4* src = reinterpret_cast<const uint4*>(P.in + b0);
      uint4 cur[4], nxt[4] = {};
#pragma unroll
      for (int k = 0; k < 4; ++k) cur[k] = __ldg(src + 4 * (STEPS - 1) + k);
      for (int step = STEPS - 1; step >= 0; --step) {
        if (step > 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) nxt[k] = __ldg(src + 4 * (step - 1) + k);
        }
#pragma unroll
        for (int k = 3; k >= 0; --k) {
          const uint32_t wq[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
#pragma unroll
          for (int j = 15; j >= 0; --j)
            G = __byte_perm(G, STV_INV_POOL, my_lut[((wq[j >> 2] >> (8 * (j & 3))) & 0xFFu) << 5]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
      }
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

// ================================================================ 1. context
struct CtxShared {
  Feed F;
  uint32_t tile_stv;
  uint32_t warp_stv[NW];
  uint32_t wv[NW][3];         // per warp: (records, column, last) of the warp
  uint32_t wpre[NW][3];       // per warp: the same over the earlier warps
  uint64_t wcnt[NW][4];       // per warp: packed value bytes per string column
  uint32_t rel[PP_MAX_COLS];  // value bytes of relative field k
  uint32_t wrd[NW];           // partial mode: per warp, 1 + its last record delimiter in the tile
  int8_t stridx[PP_MAX_COLS];
};
constexpr size_t CTX_SMEM = LUT_BYTES + 2 * TILE + sizeof(CtxShared);
constexpr int CTX_HDR = 52;  // transition vector + (records, column, last) per start state

// Per tile, from the tile's true start state: the record count, column
// offset and last terminator of the tile (ParPaRaw Sections 3.1-3.2), plus
// the value bytes per string column of the fields whose column the tile
// fixes, and per relative field of the tile's first, partial record (its
// column is only known from the scan).  The record has a slot per start
// state, as the scan composes them; only the true state's slot is filled
// and the others are zero: the scan reads a tile's slots only along the path
// from the input's start state, which enters every tile in its true state.
template <int NS>
__global__ void __launch_bounds__(NT, 3) ctx_kernel(const __grid_constant__ ParseParams P) {
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
    const uint8_t* own = tile_s + cstart;
    if (NS > 0)
      for (int k = t; k < PP_MAX_COLS; k += NT) S.rel[k] = 0;
    const uint32_t s_tile = P.s.tile_state[tile];

    // the chunk's start state, and its tags
    uint32_t G, special, special_x;
    stv_pass(w, clen, tile_s, cstart, my_lut, G, special, special_x);
    const uint32_t lane_ex = block_stv(G, S.warp_stv, &S.tile_stv);
    const uint32_t st = stv_apply(lane_ex, stv_apply(S.warp_stv[warp], s_tile));
    const Tags g = tag_chunk(st, special, special_x, P.sticky, clen, cstart, own, my_lut,
                             P.bg_next);
    if (g.inv_at < clen && st != 4)
      report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + g.inv_at, true);
    if (!P.record_end && tile + 1 == P.n_tiles && clen > 0 && cstart + clen == tile_len &&
        g.end != 4 && !((P.accept_mask >> g.end) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    if (P.s.tags)  // for the main pass: bitmaps, 1 + last terminator | end state << 16
      P.s.tags[size_t(tile) * NT + t] = make_uint4(g.fd, g.rd, g.ctrl, (g.last >> 8) | (g.end << 16));

    // (records, column, last) scanned over the warp, then over the warps
    V2 ex = chunk_v2(g);
    if (__any_sync(FULL, (ex.rec | ex.col | ex.last) != 0)) {
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const V2 o = shfl_up_v2(ex, d);
        if (lane >= d) ex = op2_32(o, ex);
      }
    }
    if (lane == 31) { S.wv[warp][0] = ex.rec; S.wv[warp][1] = ex.col; S.wv[warp][2] = ex.last; }
    {
      V2 e = shfl_up_v2(ex, 1);
      if (lane == 0) e = {0u, 0u, 0u};
      ex = e;  // exclusive within the warp
    }
    if (P.record_end) {  // partial mode: 1 + the tile's last record delimiter
      const uint32_t wm = __reduce_max_sync(FULL, g.rd ? cstart + 32u - __clz(g.rd) : 0u);
      if (lane == 0) S.wrd[warp] = wm;
    }
    __syncthreads();
    uint32_t* rec = reinterpret_cast<uint32_t*>(P.s.ctx + size_t(tile) * P.s.ctx_stride);
    if (P.record_end && t == 0) {
      uint32_t m = 0;
      for (int q = 0; q < NW; ++q) m = max(m, S.wrd[q]);
      if (m) atomicMax(P.record_end, static_cast<unsigned long long>(tile_base + m));
    }
    if (warp == 0) {
      V2 x = lane < NW ? V2{S.wv[lane][0], S.wv[lane][1], S.wv[lane][2]} : V2{0u, 0u, 0u};
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const V2 o = shfl_up_v2(x, d);
        if (lane >= d) x = op2_32(o, x);
      }
      V2 xe = shfl_up_v2(x, 1);
      if (lane == 0) xe = {0u, 0u, 0u};
      if (lane < NW) { S.wpre[lane][0] = xe.rec; S.wpre[lane][1] = xe.col; S.wpre[lane][2] = xe.last; }
      if (lane == NW - 1)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool mine = uint32_t(q) == s_tile;
          rec[1 + 3 * q] = mine ? x.rec : 0u;
          rec[2 + 3 * q] = mine ? x.col : 0u;
          rec[3 + 3 * q] = mine ? x.last : 0u;
        }
      if (lane == 0) rec[0] = S.tile_stv;
    }
    // the chunk's (records, column, last) prefix in the tile, and whether
    // the tile has control bytes: stored for the main pass
    const bool any_ctrl = __syncthreads_or(g.ctrl != 0) != 0;
    const V2 pre = op2_32(V2{S.wpre[warp][0], S.wpre[warp][1], S.wpre[warp][2]}, ex);
    if (P.s.vpre)
      P.s.vpre[size_t(tile) * NT + t] =
          make_uint2(pre.rec | ((pre.last >> 8) << 16),
                     (pre.col & 0x7FFFu) | ((pre.col & ABS32) ? 0x8000u : 0u));
    if (t == 0) P.s.tile_flags[tile] = any_ctrl ? 1u : 0u;
    if (NS > 0) {
      const uint64_t strmask = P.strmask;
      const uint32_t cmax = 63u - __clzll(static_cast<long long>(strmask));  // last string column
      const bool chain = cmax < 8;  // column masks when the string columns come early
      // value bytes per string column
      const uint32_t col0 = pre.col;  // ABS32 | column, or a relative field index
      uint64_t cnt[NSW];
#pragma unroll
      for (int k = 0; k < NSW; ++k) cnt[k] = 0;
      const uint32_t valid = range_mask(0, min(clen, g.inv_at));
      const uint32_t data = valid & ~(g.fd | g.rd | g.ctrl);
      const uint32_t T = g.fd | g.rd;
      const bool abs0 = (col0 & ABS32) != 0;
      const uint32_t c0 = col0 & ~ABS32;
      uint32_t k0 = 0xFFFFFFFFu, n0 = 0;  // the first relative segment, summed per warp below
      if (st < 4 && !chain) {
        // a walk over the chunk's fields (string columns far from the
        // record start: fewer steps than the column-by-column masks)
        bool abs = abs0;
        uint32_t col = c0, term = T, seg0 = 0;
        for (;;) {
          const uint32_t j = term ? uint32_t(__ffs(term) - 1) : 32u;
          const uint32_t n = __popc(data & range_mask(seg0, j));
          if (n && col < n_cols) {
            if (abs) {
              const int si = S.stridx[col];
              if (si >= 0) add16(cnt, si, n);
            } else if (seg0 == 0) {
              k0 = col;
              n0 = n;
            } else {
              atomicAdd(&S.rel[col], n);
            }
          }
          if (j == 32) break;
          if ((g.rd >> j) & 1u) { abs = true; col = 0; }
          else col = col < 0x7FFFFF00u ? col + 1 : col;
          seg0 = j + 1;
          term &= term - 1;
        }
      } else if (st < 4) {
        if (!abs0) {
          // fields of the tile's first, partial record: relative column
          // indices, up to this chunk's first record delimiter
          uint32_t col = c0, term = T, seg0 = 0;
          for (;;) {
            const uint32_t j = term ? uint32_t(__ffs(term) - 1) : 32u;
            const uint32_t n = __popc(data & range_mask(seg0, j));
            if (n && col < n_cols) {
              if (seg0 == 0) { k0 = col; n0 = n; }
              else atomicAdd(&S.rel[col], n);
            }
            if (j == 32 || ((g.rd >> j) & 1u)) break;
            col = col < 0x7FFFFF00u ? col + 1 : col;
            seg0 = j + 1;
            term &= term - 1;
          }
        }
        // absolute columns, one column at a time: Sc holds the starts of
        // the column's runs; T - Sc sets each run from its start up to its
        // terminator (exclusive) and clears that terminator, so the
        // terminators left out of T - Sc end the column's runs, and those
        // that are field delimiters start the next column's runs
        uint32_t Sc = (g.rd << 1) | (abs0 && c0 == 0 ? 1u : 0u);
        int si = 0;
        for (uint32_t c = 0; c <= cmax; ++c) {
          const uint32_t X = T - Sc;
          if ((strmask >> c) & 1u) {
            const uint32_t n = __popc(X & data);
            if (n) add16(cnt, si, n);
            ++si;
          }
          Sc = ((T & ~X & g.fd) << 1) | (abs0 && c0 == c + 1 ? 1u : 0u);
        }
      }
      // relative first segments (only the chunks before the tile's first
      // record delimiter have them): one shared atomic per field index
      if (__any_sync(FULL, k0 != 0xFFFFFFFFu)) {
        const uint32_t k00 = __shfl_sync(FULL, k0, 0);
        if (__all_sync(FULL, k0 == k00)) {  // the whole warp inside one field
          const uint32_t sum = __reduce_add_sync(FULL, n0);
          if (lane == 0 && sum) atomicAdd(&S.rel[k00], sum);
        } else if (k0 != 0xFFFFFFFFu && n0) {
          atomicAdd(&S.rel[k0], n0);
        }
      }
      // warp sums of the packed counters
      bool any = false;
#pragma unroll
      for (int k = 0; k < NSW; ++k) any |= cnt[k] != 0;
      if (__any_sync(FULL, any)) {
#pragma unroll
        for (int k = 0; k < NSW; ++k) {
          uint64_t v = cnt[k];
#pragma unroll
          for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
          if (lane == 0) S.wcnt[warp][k] = v;
        }
      } else if (lane == 0) {
#pragma unroll
        for (int k = 0; k < NSW; ++k) S.wcnt[warp][k] = 0;
      }
      __syncthreads();
      // the record's chars part: the true state's slot, zeros elsewhere
      uint16_t* cabs = reinterpret_cast<uint16_t*>(rec) + CTX_HDR / 2;
      uint16_t* crel = cabs + 4 * P.n_str;
      if (t < 4 * P.n_str) {
        const int s = t / P.n_str, si = t - s * P.n_str;
        uint64_t sum = 0;
        if (uint32_t(s) == s_tile) {
#pragma unroll 4
          for (int q = 0; q < NW; ++q) sum += S.wcnt[q][si >> 2];
        }
        cabs[t] = uint16_t((sum >> (16 * (si & 3))) & 0xFFFFu);
      }
      for (int k = t; k < 4 * int(n_cols); k += NT) {
        const int s = k / int(n_cols), c = k - s * int(n_cols);
        crel[k] = uint32_t(s) == s_tile ? uint16_t(S.rel[c]) : uint16_t(0);
      }
    }
    feed_next(S.F);  // the tile was last read before a barrier above
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

// Per tile, written by the scan: the tile's context, followed by the
// chars offset of the tile per string column (uint64 each).
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

// Exclusive scan over tiles of the per-start-state aggregates; every tile
// learns its true start state, record index, column and last terminator,
// then, from those, its value bytes per string column, whose exclusive
// scan gives the tile's chars offsets.
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
    if (P.dbg_withhold && blk == 0) {  // test hook: post nothing, later blocks time out
#pragma unroll
      for (int k = 0; k < 13; ++k) ex[k] = seed[k];
    } else {
      lookback_vec<13>(P.s.scan_flag_a, P.s.scan_agg_a, P.s.scan_inc_a, blk, agg, seed, ident,
                       SAggOp{}, cfg, ex);
    }
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
  const uint32_t n_cols = uint32_t(P.n_cols);
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
    if (NS > 0) {  // the tile's value bytes per string column at its true context
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

  // chars offsets: exclusive sum over tiles per string column
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
      uint64_t v[K3], x[K3], agg[K3], zero[K3], exc[K3];
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
      if (P.dbg_withhold && blk == 0) {
#pragma unroll
        for (int k = 0; k < K3; ++k) exc[k] = 0;
      } else {
        lookback_vec<K3>(P.s.scan_flag_c, P.s.scan_agg_c, P.s.scan_inc_c, blk, agg, zero, zero,
                         AddOp<K3>{}, cfg, exc);
      }
      if (lane == 0)
#pragma unroll
        for (int k = 0; k < K3; ++k) S.base[k] = exc[k];
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

// Numeric field whose bytes are not all in the tile, contain control bytes
// or need the full grammar: streaming accumulators over the value bytes.
// Returns the error bits; *out receives the value (0 for an empty field).
__device__ __forceinline__ int convert_general(const ParseParams& P, uint32_t ty, uint64_t fs,
                                            uint64_t fe, uint64_t tile_base,
                                            const uint8_t* tile_s, const uint32_t* ctrl_s,
                                            const uint32_t* my_lut, uint32_t fstate,
                                            uint64_t* out) {
  int err = 0;
  uint64_t val = 0;
  if (ty == PP_COL_FLOAT64) {
    ppn::FloatAcc acc;
    const uint32_t nd = feed_field(acc, P.in, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
    if (nd) err = acc.finish(&val);
  } else if (ty == PP_COL_TIMESTAMP) {
    ppn::TsAcc acc;
    feed_field(acc, P.in, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
    int64_t x = 0;
    err = acc.finish(&x);
    val = uint64_t(x);
  } else {
    ppn::IntAcc acc;
    const uint32_t nd = feed_field(acc, P.in, fs, fe, tile_base, tile_s, ctrl_s, my_lut, fstate);
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
  const uint8_t* tile_s;
  const uint32_t* tile_w;
  const uint32_t* ctrl_s;
  const uint16_t* cpre;
  const uint32_t* my_lut;
  bool any_ctrl;
};

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
                                             uint64_t& val) {
  val = 0;
  if (v == SLOT_DEFAULT) return 0;
  const uint32_t fsr = v >> 16, fe = v & 0xFFFFu;
  if (fsr != 0xFFFFu &&
      (!X.any_ctrl || ctrl_before(X.ctrl_s, X.cpre, fe) == ctrl_before(X.ctrl_s, X.cpre, fsr))) {
    const uint32_t L = fe - fsr;
    if (L == 0) return 0;  // empty field: the column default
    if (TY == PP_COL_TIMESTAMP) {  // five words of the tile from the field start
      const uint32_t q = fsr >> 2, sh = (fsr & 3u) * 8u;
      uint32_t x[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) x[k] = __funnelshift_r(X.tile_w[q + k], X.tile_w[q + k + 1], sh);
      int64_t t = 0;
      const int err = ppn::parse_timestamp(x, L, &t);
      val = uint64_t(t);
      return err;
    }
    const uint32_t c0 = X.tile_s[fsr];
    const uint32_t sg = (c0 == '-' || c0 == '+') ? 1u : 0u;
    const bool neg = c0 == '-';
    const int n = int(L - sg);
    const uint32_t pv = fsr + sg, q = pv >> 2, sh = (pv & 3u) * 8u;
    const uint32_t w0 = X.tile_w[q], w1 = X.tile_w[q + 1];
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
    const uint32_t x1 = __funnelshift_r(w1, X.tile_w[q + 2], sh);
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
      const uint64_t x2 = tile_load8(X.tile_w, fsr + sg + 8);
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
                         X.tile_base + fe, X.tile_base, X.tile_s, X.ctrl_s, X.my_lut,
                         X.tile_fstate, &val);
}

// Convert one row's field of a column of type TY and store it at out[rec].
template <int TY>
__device__ __forceinline__ void convert_store(const ParseParams& P, const NumCtx& X, void* out,
                                              uint64_t rec, uint32_t v) {
  uint64_t val;
  const int err = convert_field<TY>(P, v, X, val);
  if (TY == PP_COL_FLOAT64) static_cast<uint64_t*>(out)[rec] = val;
  else if (TY == PP_COL_INT64 || TY == PP_COL_TIMESTAMP) static_cast<int64_t*>(out)[rec] = int64_t(val);
  else if (TY == PP_COL_INT32) static_cast<int32_t*>(out)[rec] = int32_t(val);
  else static_cast<int8_t*>(out)[rec] = int8_t(val);
  if (err) {
    const uint32_t fsr = v >> 16;
    report(P.st, err, fsr == 0xFFFFu ? X.tile_fstart : X.tile_base + fsr, true);
  }
}

// ================================================================ 3. main
constexpr uint32_t SHORT_FIELD = 32;  // longer string fields are staged chunk-parallel
constexpr uint32_t WLIST_CAP = 512;   // terminators per warp listed in the staging buffer
constexpr uint16_t NO_FIELD = 0xFFFFu;

struct MainShared {
  Feed F;
  uint32_t tile_stv;
  uint32_t warp_stv[NW];
  uint32_t warp_rec[NW], warp_col[NW], warp_last[NW];
  uint32_t rows;             // records touched by the tile (#RD + 1)
  uint32_t col_end;          // fields of the last row closed in the tile
  uint32_t wsum[NW];
  uint32_t cstart[ppi::MAX_STR_COLS + 1];  // staging start per string column (this pass)
  uint32_t carry[ppi::MAX_STR_COLS];       // chars of earlier passes per string column
  uint64_t base[ppi::MAX_STR_COLS];        // chars offset of the tile per string column
  uint8_t coltype[PP_MAX_COLS];
  uint8_t numcol[PP_MAX_COLS];             // numeric output columns, floats first
  uint32_t n_num;
  uint16_t cpre[NT + 1];     // control bytes before chunk t (exclusive scan)
  uint16_t lk[2][NT];        // long string field (item) continuing in / starting in chunk t
};
constexpr size_t MAIN_SMEM = LUT_BYTES + 2 * TILE + STAGE_BYTES + SLOT_CAP * 4 + NT * 4 +
                             SLOT_CAP * 2 + sizeof(MainShared);



template <int NS>
__global__ void __launch_bounds__(NT, 2) main_kernel(const __grid_constant__ ParseParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin0 = smem + LUT_BYTES;  // two tile buffers
  uint8_t* stage_s = lin0 + 2 * TILE;
  uint32_t* slot_s = reinterpret_cast<uint32_t*>(stage_s + STAGE_BYTES);
  uint32_t* ctrl_s = slot_s + SLOT_CAP;
  uint16_t* pos_s = reinterpret_cast<uint16_t*>(ctrl_s + NT);  // chars end per string field
  MainShared& S = *reinterpret_cast<MainShared*>(pos_s + SLOT_CAP);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  load_lut(P, lut_s);
  for (int k = t; k < PP_MAX_COLS; k += NT) S.coltype[k] = P.coltype[k];
  if (t == 0) {
    uint32_t m = 0;
    for (uint32_t c = 0; c < uint32_t(P.n_cols); ++c)
      if (P.coltype[c] == PP_COL_FLOAT64) S.numcol[m++] = uint8_t(c);
    for (uint32_t c = 0; c < uint32_t(P.n_cols); ++c)  // the integer columns after the floats
      if (P.coltype[c] != PP_COL_SKIP && P.coltype[c] != PP_COL_STRING &&
          P.coltype[c] != PP_COL_FLOAT64)
        S.numcol[m++] = uint8_t(c);
    S.n_num = P.has_out ? m : 0u;
  }
  for (int k = t; k < ppi::MAX_STR_COLS; k += NT) S.carry[k] = 0;
  const uint32_t* my_lut = lut_s + lane;
  const uint32_t n_cols = uint32_t(P.n_cols);
  const uint32_t n_str = NS > 0 ? uint32_t(P.n_str) : 0u;
  const uint32_t rpb = max(1u, uint32_t(SLOT_CAP) / n_cols);  // rows per pass
  const bool aligned_in = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;
  uint32_t* counter = &P.s.counters[1];
  uint32_t tk = 0;  // thread 0: the next ticket
  feed_start(P, S.F, counter, aligned_in, lin0, tk);

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
    if (NS > 0 && t < int(n_str)) S.base[t] = reinterpret_cast<const uint64_t*>(pr + PRE_HDR)[t];
    uint32_t w[8];
    feed_tile(P, S.F, counter, aligned_in, lin0, tile_base, tile_len, w, tk);
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    const uint8_t* own = tile_s + cstart;

    // ---- the chunk's tags: stored by the context pass, or (without room
    // for them in the scratch) re-run here from the chunk's start state, the
    // tile's being known from the scan.  The context pass reports invalid
    // input and a bad end state.
    Tags g;
    if (P.s.tags) {
      const uint4 v = P.s.tags[size_t(tile) * NT + t];
      g = {v.x, v.y, v.z, 32u, (v.w & 0xFFFFu) << 8, v.w >> 16};
    } else {
      uint32_t G, special, special_x;
      stv_pass(w, clen, tile_s, cstart, my_lut, G, special, special_x);
      const uint32_t lane_ex = block_stv(G, S.warp_stv, &S.tile_stv);
      const uint32_t s_tile = ph.state & 0xFFu;
      const uint32_t s_chunk = stv_apply(lane_ex, stv_apply(S.warp_stv[warp], s_tile));
      g = tag_chunk(s_chunk, special, special_x, P.sticky, clen, cstart, own, my_lut, P.bg_next);
    }
    const uint32_t fd = g.fd, rd = g.rd;
    ctrl_s[t] = g.ctrl;
    const bool owns_end = last_tile && clen > 0 && cstart + clen == tile_len;
    const bool partial = P.record_end != nullptr;
    const bool virt_rd = !partial && owns_end && g.end != 4 && ((P.accept_mask >> g.end) & 1u) &&
                         !((rd >> (clen - 1)) & 1u);

    // ---- record, column and field start at the chunk start: stored by the
    // context pass with the tags, or a block scan here
    V2 pre;
    bool any_ctrl, any_virt;
    uint32_t rows, col_end_raw;  // records touched by the tile; fields of its last row
    if (P.s.vpre) {
      const uint2 pv = P.s.vpre[size_t(tile) * NT + t];
      pre = {pv.x & 0xFFFFu, (pv.y & 0x7FFFu) | ((pv.y & 0x8000u) ? ABS32 : 0u), (pv.x >> 16) << 8};
      any_ctrl = P.s.tile_flags[tile] != 0;
      V2 x = {0u, 0u, 0u};  // the tile's totals: the record's slot of the true start state
      const uint32_t s_tile = ph.state & 0xFFu;
      if (s_tile < 4) {
        const uint32_t* cr = reinterpret_cast<const uint32_t*>(P.s.ctx + size_t(tile) * P.s.ctx_stride);
        x = {cr[1 + 3 * s_tile], cr[2 + 3 * s_tile], cr[3 + 3 * s_tile]};
      }
      rows = x.rec + 1;
      if (x.col & ABS32) {
        col_end_raw = x.col & ~ABS32;
      } else {
        const uint64_t c = uint64_t(ph.col_in) + x.col;
        col_end_raw = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
      }
      any_virt = false;  // the chunk that owns the input's end closes a last record
      if (last_tile && !partial) {
        const uint32_t ot = (tile_len - 1) / CB;
        const uint4 ov = P.s.tags[size_t(tile) * NT + ot];
        const uint32_t oend = ov.w >> 16;
        any_virt = oend != 4 && ((P.accept_mask >> oend) & 1u) &&
                   !((ov.y >> (tile_len - 1 - ot * CB)) & 1u);
      }
    } else {
      V2 vi = chunk_v2(g);
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const V2 o = shfl_up_v2(vi, d);
        if (lane >= d) vi = op2_32(o, vi);
      }
      V2 lex = shfl_up_v2(vi, 1);
      if (lane == 0) lex = {0u, 0u, 0u};
      if (lane == 31) { S.warp_rec[warp] = vi.rec; S.warp_col[warp] = vi.col; S.warp_last[warp] = vi.last; }
      any_ctrl = __syncthreads_or(g.ctrl != 0) != 0;
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
        if (lane == NW - 1) {
          S.rows = x.rec + 1;
          if (x.col & ABS32) {
            S.col_end = x.col & ~ABS32;
          } else {
            const uint64_t c = uint64_t(ph.col_in) + x.col;
            S.col_end = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
          }
        }
      }
      any_virt = __syncthreads_or(virt_rd) != 0;
      pre = op2_32(V2{S.warp_rec[warp], S.warp_col[warp], S.warp_last[warp]}, lex);
      rows = S.rows;
      col_end_raw = S.col_end;
    }
    const uint64_t rec0 = ph.rec0;
    const uint32_t col_in = ph.col_in;
    const uint32_t col_end = any_virt ? n_cols : col_end_raw;
    uint32_t col0;
    if (pre.col & ABS32) {
      col0 = pre.col & ~ABS32;
    } else {
      const uint64_t c = uint64_t(col_in) + pre.col;
      col0 = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
    }
    // the field open at the tile start: global start and DFA state there
    const uint64_t tile_fstart = ph.last1;
    const uint32_t tile_fstate = ph.last1 ? (ph.state >> 8) & 0xFFu : uint32_t(P.start_state);
    const uint32_t fs_tile = tile_fstart >= tile_base ? uint32_t(tile_fstart - tile_base) : 0xFFFFu;
    const uint32_t fs0 = pre.last ? (pre.last >> 8) : fs_tile;  // field open at the chunk start
    const uint32_t rl0 = pre.rec;
    const uint32_t term_all = fd | rd;
    const bool owns_tail = clen > 0 && cstart + clen == tile_len;
    // terminators per chunk (plus the virtual RD that closes the input),
    // their prefix in the warp and the warp's count
    const uint32_t nterm = __popc(term_all) + (virt_rd ? 1u : 0u);
    uint32_t tincl = nterm;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, tincl, d);
      if (lane >= d) tincl += o;
    }
    const uint32_t tbase = tincl - nterm, wn = __shfl_sync(FULL, tincl, 31);
    if (any_ctrl) {  // control bytes before each chunk: O(1) value-byte counts
      const uint32_t nc = __popc(g.ctrl);
      uint32_t xi = nc;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, xi, d);
        if (lane >= d) xi += o;
      }
      if (lane == 31) S.wsum[warp] = xi;
      __syncthreads();
      if (warp == 0) {
        const uint32_t v = lane < NW ? S.wsum[lane] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int d = 1; d < NW; d <<= 1) {
          const uint32_t o = __shfl_up_sync(FULL, x, d);
          if (lane >= d) x += o;
        }
        __syncwarp();
        if (lane < NW) S.wsum[lane] = x - v;
        if (lane == NW - 1) S.cpre[NT] = uint16_t(x);
      }
      __syncthreads();
      S.cpre[t] = uint16_t(S.wsum[warp] + xi - nc);
    }

    const NumCtx X = {tile_base, tile_fstart, tile_fstate, tile_s, tile_w, ctrl_s, S.cpre, my_lut,
                      any_ctrl};
    const uint32_t rec_lim =  // records of the tile the outputs have room for
        P.rec_cap > rec0 ? uint32_t(min(P.rec_cap - rec0, uint64_t(0xFFFFFFFFu))) : 0u;

    // ---- fields -> (column, row) slots, in passes of rows
    {
      for (uint32_t lo = 0; lo < rows; lo += rpb) {
        const uint32_t hi = min(rows, lo + rpb), nr = hi - lo;
        if (NS > 0) { S.lk[0][t] = NO_FIELD; S.lk[1][t] = NO_FIELD; }
        if (wn <= WLIST_CAP) {
          // the warp's terminators in input order (tile position | RD << 15),
          // then a lane per field: row and column from a ballot of the RDs
          uint16_t* const wl = reinterpret_cast<uint16_t*>(stage_s) + warp * WLIST_CAP;
          {
            uint32_t m = term_all, i = tbase;
            while (m) {
              const uint32_t j = __ffs(m) - 1;
              m &= m - 1;
              wl[i++] = uint16_t((cstart + j) | (((rd >> j) & 1u) << 15));
            }
            if (virt_rd) wl[i] = uint16_t(tile_len | 0x8000u);
          }
          __syncwarp();
          // row, column and field start before the batch's first field
          uint32_t crow = __shfl_sync(FULL, rl0, 0), ccol = __shfl_sync(FULL, col0, 0),
                   cfs = __shfl_sync(FULL, fs0, 0);
          const uint32_t lt = (1u << lane) - 1u;
          for (uint32_t b0 = 0; b0 < wn; b0 += 32) {
            const uint32_t k = b0 + uint32_t(lane);
            const uint32_t ent = k < wn ? uint32_t(wl[k]) : 0u;
            const uint32_t e = ent & 0x7FFFu;
            const bool isrd = (ent >> 15) != 0;
            const uint32_t pe = __shfl_up_sync(FULL, e, 1);
            const uint32_t fs = lane == 0 ? cfs : pe + 1u;
            const uint32_t rdm = __ballot_sync(FULL, isrd);
            const uint32_t below = rdm & lt;
            const uint32_t rl = crow + __popc(below);
            const uint32_t col = below ? uint32_t(lane) - (32u - __clz(below))
                                       : min(ccol + uint32_t(lane), 0x7FFFFF00u);
            if (k < wn) {
              const bool in_pass = rl - lo < nr;
              if (in_pass && col < n_cols) slot_s[col * nr + (rl - lo)] = (fs << 16) | e;
              if (isrd && col != n_cols - 1) {
                if (lo == 0) report(P.st, PP_ERR_COLCOUNT, tile_base + e, true);
                if (in_pass)  // missing fields take the column default
                  for (uint32_t c = col + 1; c < n_cols; ++c) slot_s[c * nr + (rl - lo)] = SLOT_DEFAULT;
              }
            }
            const uint32_t nin = min(32u, wn - b0);
            crow += __popc(rdm);
            ccol = rdm ? (nin - 1u) - (31u - __clz(rdm)) : min(ccol + nin, 0x7FFFFF00u);
            cfs = __shfl_sync(FULL, e, nin - 1) + 1u;
          }
          // the field still open at the tile end (its value bytes are staged)
          if (NS > 0 && owns_tail && !any_virt && crow - lo < nr && ccol < n_cols)
            slot_s[ccol * nr + (crow - lo)] = (cfs << 16) | tile_len;
        } else {  // each lane walks its chunk's fields
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
            const bool in_pass = rl - lo < nr;
            if (in_pass && col < n_cols) slot_s[col * nr + (rl - lo)] = (fs << 16) | e;
            if (isrd) {
              if (col != n_cols - 1) {
                if (lo == 0) report(P.st, PP_ERR_COLCOUNT, tile_base + e, true);
                if (in_pass)  // missing fields take the column default
                  for (uint32_t c = col + 1; c < n_cols; ++c) slot_s[c * nr + (rl - lo)] = SLOT_DEFAULT;
              }
              ++rl;
              col = 0;
            } else {
              col = col < 0x7FFFFF00u ? col + 1 : col;
            }
            fs = e + 1;
          }
          // the field still open at the tile end (its value bytes are staged)
          if (NS > 0 && owns_tail && !any_virt && rl - lo < nr && col < n_cols)
            slot_s[col * nr + (rl - lo)] = (fs << 16) | tile_len;
        }
        __syncthreads();
        const uint32_t ngr = (nr + 31) / 32;
        if (lo == 0 && P.s.tags) {  // the next tile's stored tags and prefixes, towards L2
          const uint32_t nt = S.F.tile[S.F.cur ^ 1u];  // taken before the barrier above
          if (nt < P.n_tiles) {
            if ((t & 7) == 0) prefetch_l2(P.s.tags + size_t(nt) * NT + t);
            if ((t & 15) == 0) prefetch_l2(P.s.vpre + size_t(nt) * NT + t);
          }
        }

        if (NS > 0 && n_str) {
          // ---- string fields: value bytes -> chars positions (block scan
          // over the column-major items), then staging copies
          const uint32_t n_items = n_str * nr;
          const uint32_t per = (n_items + NT - 1) / NT;  // <= SLOT_CAP / NT
          const uint32_t k0 = min(n_items, uint32_t(t) * per), k1 = min(n_items, k0 + per);
          // value bytes per field (into pos_s for now), long fields mark their chunks
          uint32_t mysum = 0;
          {
            uint32_t si = k0 / nr, r = k0 - si * nr;
            for (uint32_t k = k0; k < k1; ++k) {
              uint32_t len = 0;
              const uint32_t c = P.strcol[si];
              const uint32_t row = lo + r;
              const bool closed = (row > 0 || c >= col_in) && (row + 1 < rows || c < col_end);
              const bool open = row + 1 == rows && c == col_end && !any_virt;
              if (closed || open) {
                const uint32_t v = slot_s[c * nr + r];
                if (v != SLOT_DEFAULT) {
                  const bool before = (v >> 16) == 0xFFFFu;
                  const uint32_t a0 = before ? 0u : (v >> 16), e = v & 0xFFFFu;
                  len = (e - a0) - (any_ctrl ? ctrl_before(ctrl_s, S.cpre, e) -
                                                   ctrl_before(ctrl_s, S.cpre, a0) : 0u);
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
          __syncthreads();
          if (warp == 0) {
            const uint32_t v = lane < NW ? S.wsum[lane] : 0u;
            uint32_t x = v;
#pragma unroll
            for (int d = 1; d < NW; d <<= 1) {
              const uint32_t o = __shfl_up_sync(FULL, x, d);
              if (lane >= d) x += o;
            }
            __syncwarp();
            if (lane < NW) S.wsum[lane] = x - v;
            if (lane == NW - 1) S.cstart[n_str] = x;
          }
          __syncthreads();
          {  // lengths -> chars end positions (inclusive prefix)
            uint32_t run = S.wsum[warp] + xi - mysum;
            uint32_t si = k0 / nr, r = k0 - si * nr;
            for (uint32_t k = k0; k < k1; ++k) {
              if (r == 0) S.cstart[si] = run;
              run += pos_s[k];
              pos_s[k] = uint16_t(run);
              if (++r == nr) { r = 0; ++si; }
            }
          }
          __syncthreads();
          // staging: a lane per short field; long fields chunk-parallel,
          // each thread copying its chunk's part of the (at most two) long
          // fields that cover it
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
              const uint32_t v = slot_s[c * nr + rr];
              const uint32_t a0 = (v >> 16) == 0xFFFFu ? 0u : (v >> 16), e = v & 0xFFFFu;
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
              const uint32_t v = slot_s[P.strcol[ksi] * nr + (k - ksi * nr)];
              const uint32_t a0 = (v >> 16) == 0xFFFFu ? 0u : (v >> 16), e = v & 0xFFFFu;
              const uint32_t p0 = max(a0, cstart), p1 = min(e, cstart + clen);
              const uint32_t c_a0 = any_ctrl ? ctrl_before(ctrl_s, S.cpre, a0) : 0u;
              const uint32_t c_e = any_ctrl ? ctrl_before(ctrl_s, S.cpre, e) : 0u;
              const uint32_t c_p0 = any_ctrl ? ctrl_before(ctrl_s, S.cpre, p0) : 0u;
              const uint32_t len = (e - a0) - (c_e - c_a0);
              uint32_t dst = pos_s[k] - len + (p0 - a0) - (c_p0 - c_a0);
              const uint32_t cm = g.ctrl & range_mask(p0 - cstart, p1 - cstart);
              if (!cm) {
                for (uint32_t p = p0; p < p1; ++p) stage_s[dst++] = tile_s[p];
              } else {
                for (uint32_t p = p0; p < p1; ++p)
                  if (!((cm >> (p - cstart)) & 1u)) stage_s[dst++] = tile_s[p];
              }
            }
          }
        }

        // ---- numbers: a lane per (numeric column, row) slot, the slots of
        // the numeric columns taken column by column, 32 to a warp; columns
        // of one type are adjacent, so a warp mostly runs one conversion
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
            if (r >= rec_lim) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
            const uint32_t v = slot_s[c * nr + (r - lo)];
            void* const out = P.typed[c];
            const uint64_t rec = rec0 + r;
            switch (S.coltype[c]) {
              case PP_COL_FLOAT64: convert_store<PP_COL_FLOAT64>(P, X, out, rec, v); break;
              case PP_COL_INT64: convert_store<PP_COL_INT64>(P, X, out, rec, v); break;
              case PP_COL_TIMESTAMP: convert_store<PP_COL_TIMESTAMP>(P, X, out, rec, v); break;
              case PP_COL_INT32: convert_store<PP_COL_INT32>(P, X, out, rec, v); break;
              default: convert_store<PP_COL_INT8>(P, X, out, rec, v); break;
            }
          }
        }
        __syncthreads();
        if (NS > 0 && n_str && P.has_out) {
          // Arrow offsets of the string fields closed in this pass
          uint32_t si = 0, gi = uint32_t(warp);
          while (gi >= ngr && si < n_str) { gi -= ngr; ++si; }
          for (; si < n_str; gi += NW) {
            while (gi >= ngr && si < n_str) { gi -= ngr; ++si; }
            if (si >= n_str) break;
            const uint32_t r = lo + gi * 32 + lane;
            const uint32_t c = P.strcol[si];
            if (r >= hi || (r == 0 && c < col_in) || (r + 1 == rows && c >= col_end)) continue;
            const uint64_t rec = rec0 + r;
            if (rec >= P.rec_cap) { report(P.st, PP_ERR_CAPACITY, 0, false); continue; }
            const uint64_t off = S.base[si] + S.carry[si] + (pos_s[si * nr + (r - lo)] - S.cstart[si]);
            if (off > 0x7FFFFFFFull || off > P.chars_cap[si]) report(P.st, PP_ERR_CAPACITY, 0, false);
            else P.offsets[si][rec + 1] = int32_t(off);
          }
          // staged chars -> HBM, 16-byte aligned stores
          for (uint32_t si = 0; si < n_str; ++si) {
            uint32_t len = S.cstart[si + 1] - S.cstart[si];
            if (!len) continue;
            const uint64_t gb = S.base[si] + S.carry[si];
            if (gb + len > P.chars_cap[si]) {
              if (t == 0) report(P.st, PP_ERR_CAPACITY, 0, false);
              len = gb >= P.chars_cap[si] ? 0u : uint32_t(P.chars_cap[si] - gb);
            }
            uint8_t* gp = P.chars[si] + gb;
            const uint32_t sp = S.cstart[si];
            const uint32_t head = min(len, uint32_t((16u - (reinterpret_cast<uintptr_t>(gp) & 15u)) & 15u));
            const uint32_t nvec = (len - head) >> 4;
            const uint32_t tail0 = head + (nvec << 4);
            if (uint32_t(t) < head) gp[t] = stage_s[sp + t];
            const uint32_t src0 = sp + head;
            const uint32_t sh = (src0 & 3u) * 8u;
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(stage_s + (src0 & ~3u));
            uint4* gv = reinterpret_cast<uint4*>(gp + head);
            for (uint32_t v = t; v < nvec; v += NT) {
              const uint32_t* q = sw + 4 * v;
              const uint32_t a0 = q[0], a1 = q[1], a2 = q[2], a3 = q[3], a4 = q[4];
              uint4 o;
              o.x = __funnelshift_r(a0, a1, sh);
              o.y = __funnelshift_r(a1, a2, sh);
              o.z = __funnelshift_r(a2, a3, sh);
              o.w = __funnelshift_r(a3, a4, sh);
              __stcs(gv + v, o);
            }
            if (tail0 + t < len) gp[tail0 + t] = stage_s[sp + tail0 + t];
          }
        }
        __syncthreads();
        if (NS > 0 && t < int(n_str)) S.carry[t] += S.cstart[t + 1] - S.cstart[t];
      }
    }
    __syncthreads();
    if (t < int(n_str)) {
      if (last_tile) P.st->chars_len[P.strcol[t]] = S.base[t] + S.carry[t];
      S.carry[t] = 0;
    }
    if (owns_end) P.st->n_records = rec0 + (rows - 1) + (virt_rd ? 1u : 0u);
    feed_next(S.F);  // the tile was last read before a barrier above
  }
  feed_finish(S.F);
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
// Zero the tile counters and the scan's look-back flags; initialise the
// status and offsets[c][0] = 0 for every string column.
__global__ void parse_init_kernel(ParseParams P) {
  const ppi::ParseScratch& s = P.s;
  const uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = i0; i < s.n_scan_blocks; i += stride) { s.scan_flag_a[i] = 0; s.scan_flag_c[i] = 0; }
  for (uint32_t i = i0; i < s.n_tstate_blocks; i += stride) s.tstate_words[i] = 0;
  if (i0 < 4) s.counters[i0] = 0;
  if (i0 == 0) {
    pp_status* st = P.st;
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

struct Occ { int ctx = 1, main = 1, n_sm = 0; };

// Per device: the SM count, the dynamic shared-memory attributes of the two
// big tile passes and their resident blocks per SM.
template <int NS>
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
    if ((r = cudaFuncSetAttribute(ctx_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(CTX_SMEM))) != cudaSuccess)
      return r;
    if ((r = cudaFuncSetAttribute(main_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(MAIN_SMEM))) != cudaSuccess)
      return r;
    int b = 0;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, ctx_kernel<NS>, NT, CTX_SMEM)) !=
        cudaSuccess)
      return r;
    o.ctx = b > 0 ? b : 1;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, main_kernel<NS>, NT, MAIN_SMEM)) !=
        cudaSuccess)
      return r;
    o.main = b > 0 ? b : 1;
    occ[d] = o;
    return cudaSuccess;
  });
  *out = &occ[dev];
  return e;
}

template <int NS>
cudaError_t launch_ns(const ParseParams& p, cudaStream_t stream) {
  Occ* po = nullptr;
  cudaError_t e = parse_setup<NS>(&po);
  if (e != cudaSuccess) return e;
  const Occ& occ = *po;
  const bool timed = ppi::stage_begin();
  if (timed) ppi::stage_mark(0, stream);
  parse_init_kernel<<<std::max<uint32_t>(1, std::min<uint32_t>((p.s.n_scan_blocks + 255) / 256, 1024)),
                      256, 0, stream>>>(p);
  if (timed) ppi::stage_mark(1, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) {
    const uint32_t gv = uint32_t(std::min<uint64_t>((p.n_tiles + TV_NT / 32 - 1) / (TV_NT / 32),
                                                    uint64_t(occ.n_sm) * 6));
    tile_stv_kernel<<<gv, TV_NT, LUT_BYTES, stream>>>(p);
  }
  if (timed) ppi::stage_mark(2, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) tile_state_kernel<<<p.s.n_tstate_blocks, TS_NT, 0, stream>>>(p);
  if (timed) ppi::stage_mark(3, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const uint32_t g1 = uint32_t(std::min<uint64_t>(std::max<uint32_t>(p.n_tiles, 1),
                                                  uint64_t(occ.n_sm) * occ.ctx));
  if (p.n_tiles) ctx_kernel<NS><<<g1, NT, CTX_SMEM, stream>>>(p);
  if (timed) ppi::stage_mark(4, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) scan_kernel<NS><<<p.s.n_scan_blocks, SCAN_NT, 0, stream>>>(p);
  if (timed) ppi::stage_mark(5, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const uint32_t g3 = uint32_t(std::min<uint64_t>(std::max<uint32_t>(p.n_tiles, 1),
                                                  uint64_t(occ.n_sm) * occ.main));
  if (p.n_tiles) main_kernel<NS><<<g3, NT, MAIN_SMEM, stream>>>(p);
  if (timed) ppi::stage_mark(6, stream);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
uint32_t ctx_stride_of(int ns, int n_cols) {
  const size_t b = CTX_HDR + (ns > 0 ? 8 * size_t(ns) + 8 * size_t(n_cols) : 0);
  return uint32_t((b + 15) & ~size_t(15));
}
uint32_t pre_stride_of(int ns) { return uint32_t(PRE_HDR + 8 * (ns > 0 ? ns : 0)); }

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
    int b = 0;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fields_kernel, NT, FIELDS_SMEM)) !=
        cudaSuccess)
      return r;
    occ_of[d] = b > 0 ? b : 1;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int occ = occ_of[dev];
  parse_init_kernel<<<1, 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_tiles) {
    const uint32_t gv = uint32_t(std::min<uint64_t>((p.n_tiles + TV_NT / 32 - 1) / (TV_NT / 32),
                                                    uint64_t(n_sm) * 6));
    tile_stv_kernel<<<gv, TV_NT, LUT_BYTES, stream>>>(p);
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

int parse_ns_width(int n_str) {
  if (n_str <= 0) return 0;
  if (n_str <= 4) return 4;
  if (n_str <= 8) return 8;
  return 16;
}

// layout: counters | scan flags (records, chars) | scan payloads (2 x 13
// words per scan block; 2 x ns words per scan block) | ctx records | pre
// records
size_t parse_scratch_bytes(uint32_t n, int ns, int n_cols, bool tags) {
  const uint32_t nb = (n + SCAN_TILES - 1) / SCAN_TILES;
  const uint32_t nt = (n + TS_TILES - 1) / TS_TILES;
  const int k3 = ns > 0 ? ns : 1;
  return 256 + 2 * align256(size_t(nb) * 4) + 2 * align256(size_t(nb) * 13 * 8) +
         2 * align256(size_t(nb) * k3 * 8) + align256(size_t(n) * ctx_stride_of(ns, n_cols)) +
         align256(size_t(n) * pre_stride_of(ns)) + align256(size_t(n) * 4) + align256(n) +
         align256(size_t(nt) * 8) + align256(n) + (tags ? align256(size_t(n) * NT * 24) : 0);
}

void parse_scratch_carve(void* base, uint32_t n, int ns, int n_cols, bool tags, ParseScratch* o) {
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
  o->pre = p; p += align256(size_t(n) * pre_stride_of(ns));
  o->tile_stv = reinterpret_cast<uint32_t*>(p); p += align256(size_t(n) * 4);
  o->tile_state = p; p += align256(n);
  o->tstate_words = reinterpret_cast<unsigned long long*>(p);
  o->n_tstate_blocks = (n + TS_TILES - 1) / TS_TILES;
  p += align256(size_t(o->n_tstate_blocks) * 8);
  o->tile_flags = p; p += align256(n);
  o->tags = tags ? reinterpret_cast<uint4*>(p) : nullptr;
  if (tags) p += size_t(n) * NT * 16;
  o->vpre = tags ? reinterpret_cast<uint2*>(p) : nullptr;
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
