// pp_parse: single-pass DFA-based parsing of delimiter-separated input into
// Arrow-style columns on sm_103a.
//
// Persistent CTAs of 512 threads take 16 KiB tiles in order from an atomic
// counter.  Per tile:
//   S1  the tile arrives in shared memory by a 1-D bulk copy (TMA engine),
//       issued while the previous tile was being processed; HBM input is
//       read exactly once.  Each thread moves its 32-byte chunk into
//       registers and writes it back word-interleaved (word k of thread t at
//       k*512+t), so that every later per-thread byte access hits the
//       thread's own bank.
//   S2  each thread runs the multi-instance DFA over its chunk (ParPaRaw
//       Section 3.1, Figure 2): the state-transition vector of all live
//       states sits in one register, one byte per state, and each input
//       byte composes it with the byte's symbol-group transition by one
//       byte-permute — the row-per-symbol-group transition table of ParPaRaw
//       Section 5 (Table 1), fetched from a per-lane replicated shared-memory
//       LUT so the lookup never bank-conflicts.
//   S3  warp shuffles and a block pass compose the vectors; a single-pass
//       decoupled look-back over tiles gives the tile's exclusive composite
//       prefix, seeded with the identity (ParPaRaw Section 3.1).
//   S5  each thread re-runs ONE DFA from its true start state over the
//       chunk's non-background bytes only and builds the three bitmap
//       indexes (record delimiter, field delimiter, control; Section 3.1).
//   S6  record counts (POPCNT) and absolute/relative column offsets
//       (ParPaRaw Section 3.2, Figure 4) are scanned across the block and the
//       tiles (second look-back), then the per-string-column value-byte
//       counts (third look-back) place the tile in every chars buffer.
//   S7  value bytes of string columns are compacted per column into shared
//       memory and leave as contiguous 16-byte stores (the column
//       partitioning of ParPaRaw Section 3.3 done as stream compaction).
//   S8  every closed field is entered in a column-major (column, record)
//       slot table; one lane per field then writes Arrow offsets or converts
//       the number (ParPaRaw Section 3.3, thread-exclusive level), so a warp
//       works on one column — one type — and its stores are coalesced.
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
constexpr uint64_t ABS64 = 1ull << 63;
constexpr uint32_t ABS32 = 1u << 31;
constexpr uint32_t SLOT_ABSENT = 0xFFFFFFFEu;  // field not closed in this tile
constexpr uint32_t SLOT_DEFAULT = 0xFFFFFFFDu; // missing field: column default
constexpr uint32_t WAIT_LIMIT = 1u << 24;      // bounded mbarrier polls

struct Shared {
  uint64_t bar;              // bulk-copy completion
  uint32_t tile, next_tile;
  uint32_t issued;           // a bulk copy is in flight into lin_s
  uint32_t parity;
  uint32_t stv_prefix;
  uint32_t rows;             // records touched by the tile (#RD + 1)
  uint32_t warp_stv[NW];
  uint32_t warp_rec[NW], warp_col[NW], warp_last[NW];
  uint64_t lb2[4];
  uint64_t wcnt[NW][4];
  uint64_t base[ppi::MAX_STR_COLS];
  uint32_t total[ppi::MAX_STR_COLS];
  uint32_t R[ppi::MAX_STR_COLS];
  int8_t stridx[PP_MAX_COLS];
  uint8_t coltype[PP_MAX_COLS];
  uint8_t outcol[PP_MAX_COLS];  // columns that produce output, in order
  uint32_t n_out;
};

constexpr size_t SMEM_BYTES = LUT_BYTES + 2 * TILE + STAGE_BYTES + SLOT_CAP * 4 + NT * 4 +
                              sizeof(Shared);

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

// Tile-level version of the same operator on (rec, col, last pos+1, state).
struct Op2 {
  __device__ void operator()(const uint64_t (&a)[4], const uint64_t (&b)[4],
                             uint64_t (&o)[4]) const {
    o[0] = a[0] + b[0];
    o[1] = (b[1] & ABS64) ? b[1] : ((a[1] & ABS64) | ((a[1] & ~ABS64) + b[1]));
    const bool hb = b[2] != 0;
    o[2] = hb ? b[2] : a[2];
    o[3] = hb ? b[3] : a[3];
  }
};
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

// byte p of the tile in the word-interleaved layout
__device__ __forceinline__ uint32_t tile_byte(const uint8_t* tile_s, uint32_t p) {
  return tile_s[((((p & 31u) >> 2) * NT + (p >> 5)) << 2) | (p & 3u)];
}
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

// Issue the bulk copy of tile `tile` into the landing buffer (thread 0).
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

template <int NS>
__global__ void __launch_bounds__(NT, 2) parse_kernel(const __grid_constant__ ParseParams P) {
  constexpr int NSW = NS > 0 ? (NS + 3) / 4 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* lin_s = smem + LUT_BYTES;            // bulk-copy landing buffer
  uint8_t* tile_s = lin_s + TILE;               // word-interleaved tile
  uint8_t* stage_s = tile_s + TILE;
  uint32_t* slot_s = reinterpret_cast<uint32_t*>(stage_s + STAGE_BYTES);
  uint32_t* ctrl_s = slot_s + SLOT_CAP;
  Shared& S = *reinterpret_cast<Shared*>(ctrl_s + NT);
  uint32_t* tile_w = reinterpret_cast<uint32_t*>(tile_s);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int k = t; k < 256 * 32; k += NT) lut_s[k] = P.lut[k >> 5];
  for (int k = t; k < PP_MAX_COLS; k += NT) {
    S.stridx[k] = P.stridx[k];
    S.coltype[k] = P.coltype[k];
  }
  const uint32_t* my_lut = lut_s + lane;
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t n_cols = uint32_t(P.n_cols);
  const bool aligned_in = (reinterpret_cast<uintptr_t>(P.in) & 15) == 0;

  if (t == 0) {
    uint32_t k = 0;
    for (uint32_t c = 0; c < n_cols; ++c)
      if (P.coltype[c] != PP_COL_SKIP) S.outcol[k++] = uint8_t(c);
    S.n_out = k;
    mbar_init(&S.bar, 1);
    S.parity = 0;
    const uint32_t tile = atomicAdd(P.s.tile_counter, 1u);
    S.tile = tile;
    S.issued = issue_tile(P, tile, aligned_in, lin_s, &S.bar);
  }
  __syncthreads();

  for (;;) {
    const uint32_t tile = S.tile;
    if (tile >= P.n_tiles) break;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    const bool last_tile = tile + 1 == P.n_tiles;

    // ---------------------------------------------------------------- S1
    const uint32_t bulk = S.issued ? (tile_len & ~15u) : 0u;
    if (S.issued) {
      if (!mbar_wait_bounded(&S.bar, S.parity, WAIT_LIMIT)) {
        if (t == 0) report(P.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
        mbar_wait_bounded(&S.bar, S.parity, WAIT_LIMIT);
      }
    }
    if (bulk < tile_len) {  // ragged tail / unaligned input: plain loads
      for (uint32_t k = bulk + t; k < tile_len; k += NT) lin_s[k] = P.in[tile_base + k];
      __syncthreads();
    }
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    uint32_t w[8];
    {
      const uint4* src = reinterpret_cast<const uint4*>(lin_s + cstart);
      const int sw = (t >> 2) & 1;  // alternate read order: conflict-free 16-byte reads
      const uint4 x = src[sw], y = src[sw ^ 1];
      const uint4 lo = sw ? y : x, hi = sw ? x : y;
      w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
      w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
#pragma unroll
      for (int k = 0; k < 8; ++k) tile_w[k * NT + t] = w[k];
    }
    __syncthreads();
    if (t == 0) {  // prefetch the next tile into the (now free) landing buffer
      if (S.issued) S.parity ^= 1u;
      const uint32_t nt = atomicAdd(P.s.tile_counter, 1u);
      S.next_tile = nt;
      S.issued = issue_tile(P, nt, aligned_in, lin_s, &S.bar);
    }

    // ---------------------------------------------------------------- S2
    uint32_t G = STV_ID, special = 0;
    if (clen == CB) {
#pragma unroll
      for (int j = CB - 1; j >= 0; --j) {
        const uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        const uint32_t e = my_lut[b << 5];
        G = __byte_perm(G, STV_INV_POOL, e);   // G := G o delta_group(b)
        special = __funnelshift_l(e, special, 1);
      }
    } else {
      for (int j = int(clen) - 1; j >= 0; --j) {
        const uint32_t e = my_lut[tile_byte(tile_s, cstart + j) << 5];
        G = __byte_perm(G, STV_INV_POOL, e);
        special = __funnelshift_l(e, special, 1);
      }
    }

    // ---------------------------------------------------------------- S3
    uint32_t inc = G;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, inc, d);
      if (lane >= d) inc = stv_compose(o, inc);
    }
    uint32_t lane_ex = __shfl_up_sync(FULL, inc, 1);
    if (lane == 0) lane_ex = STV_ID;
    if (lane == 31) S.warp_stv[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const uint32_t v = lane < NW ? S.warp_stv[lane] : STV_ID;
      uint32_t wi = v;
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, wi, d);
        if (lane >= d) wi = stv_compose(o, wi);
      }
      uint32_t wex = __shfl_up_sync(FULL, wi, 1);
      if (lane == 0) wex = STV_ID;
      const uint32_t agg = __shfl_sync(FULL, wi, NW - 1);
      if (lane < NW) S.warp_stv[lane] = wex;
      const uint32_t pre = lookback_word(
          P.s.lb1, tile, agg, STV_ID, STV_ID,
          [](uint32_t a, uint32_t b) { return stv_compose(a, b); }, cfg);
      if (lane == 0) S.stv_prefix = pre;
    }
    __syncthreads();
    uint32_t s = stv_apply(S.stv_prefix, P.start_state);
    s = stv_apply(S.warp_stv[warp], s);
    s = stv_apply(lane_ex, s);
    const uint32_t s_chunk = s;

    // ---------------------------------------------------------------- S5
    const uint8_t* own = tile_s + 4 * t;  // byte j of own chunk: own[(j>>2)*4*NT + (j&3)]
    uint32_t fd = 0, rd = 0, ctrl = 0, inv_at = 32, last_term = 0;
    if (s == 4) {
      inv_at = 0;
    } else {
      uint32_t m = special & range_mask(0, clen);
      uint32_t prev = 0;
      while (m) {
        const uint32_t j = __ffs(m) - 1;
        m &= m - 1;
        if (j > prev) {  // a run of background bytes: one idempotent transition
          const uint32_t s1 = (P.bg_next >> (4 * s)) & 0xFu;
          if (s1 == 4) { inv_at = prev; s = 4; break; }
          s = s1;
        }
        const uint32_t byte = own[(j >> 2) * (4 * NT) + (j & 3)];
        const uint32_t e = my_lut[byte << 5];
        const uint32_t nx = (e >> (4 * s)) & 0xFu;
        if (nx == 4) { inv_at = j; s = 4; break; }
        const uint32_t tg = (e >> (20 + 2 * s)) & 3u;
        const uint32_t bit = 1u << j;
        fd |= tg == PP_TAG_FD ? bit : 0u;
        rd |= tg == PP_TAG_RD ? bit : 0u;
        ctrl |= tg == PP_TAG_CTRL ? bit : 0u;
        if (tg == PP_TAG_FD || tg == PP_TAG_RD) last_term = ((cstart + j + 1) << 8) | nx;
        s = nx;
        prev = j + 1;
      }
      if (s != 4 && prev < clen) {
        const uint32_t s1 = (P.bg_next >> (4 * s)) & 0xFu;
        if (s1 == 4) { inv_at = prev; s = 4; } else { s = s1; }
      }
    }
    const uint32_t valid = range_mask(0, min(clen, inv_at));
    const uint32_t data = valid & ~(fd | rd | ctrl);
    ctrl_s[t] = ctrl;
    if (inv_at < clen && s_chunk != 4)
      report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + inv_at, true);
    const bool owns_end = last_tile && clen > 0 && cstart + clen == tile_len;
    if (owns_end && s != 4 && !((P.accept_mask >> s) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    const bool virt_rd = owns_end && s != 4 && ((P.accept_mask >> s) & 1u) &&
                         !((rd >> (clen - 1)) & 1u);

    // --------------------------------------------------------------- S6a
    V2 my;
    my.rec = __popc(rd);
    if (rd) {
      const uint32_t hi = 31 - __clz(rd);
      my.col = ABS32 | uint32_t(__popc(hi == 31 ? 0u : (fd >> (hi + 1))));
    } else {
      my.col = uint32_t(__popc(fd));
    }
    my.last = last_term;
    V2 vi = my;
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
      V2 w2 = lane < NW ? V2{S.warp_rec[lane], S.warp_col[lane], S.warp_last[lane]} : V2{0u, 0u, 0u};
      V2 wi = w2;
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const V2 o = shfl_up_v2(wi, d);
        if (lane >= d) wi = op2_32(o, wi);
      }
      V2 wex = shfl_up_v2(wi, 1);
      if (lane == 0) wex = {0u, 0u, 0u};
      const V2 agg = {__shfl_sync(FULL, wi.rec, NW - 1), __shfl_sync(FULL, wi.col, NW - 1),
                      __shfl_sync(FULL, wi.last, NW - 1)};
      if (lane < NW) { S.warp_rec[lane] = wex.rec; S.warp_col[lane] = wex.col; S.warp_last[lane] = wex.last; }
      const uint64_t a4[4] = {agg.rec, ((agg.col & ABS32) ? ABS64 : 0ull) | (agg.col & ~ABS32),
                              agg.last ? tile_base + (agg.last >> 8) : 0ull, agg.last & 0xFFu};
      const uint64_t seed[4] = {0ull, ABS64, 0ull, 0ull};
      const uint64_t ident[4] = {0ull, 0ull, 0ull, 0ull};
      uint64_t ex[4];
      lookback_vec<4>(P.s.lb2_flag, P.s.lb2_agg, P.s.lb2_inc, tile, a4, seed, ident, Op2{}, cfg, ex);
      if (lane == 0) {
        S.lb2[0] = ex[0]; S.lb2[1] = ex[1]; S.lb2[2] = ex[2]; S.lb2[3] = ex[3];
        S.rows = agg.rec + 1;
      }
    }
    __syncthreads();
    const V2 pre = op2_32(V2{S.warp_rec[warp], S.warp_col[warp], S.warp_last[warp]}, lex);
    const uint64_t tile_rec0 = S.lb2[0];
    const uint64_t rec0 = tile_rec0 + pre.rec;
    uint32_t col0;
    if (pre.col & ABS32) {
      col0 = pre.col & ~ABS32;
    } else {
      const uint64_t c = (S.lb2[1] & ~ABS64) + pre.col;
      col0 = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
    }
    uint64_t fstart0;
    if (pre.last) fstart0 = tile_base + (pre.last >> 8);
    else fstart0 = S.lb2[2];  // 0 when no terminator precedes the chunk
    // start (global) and DFA state of the field holding tile byte 0
    const uint64_t tile_fstart = S.lb2[2];
    const uint32_t tile_fstate = S.lb2[2] ? uint32_t(S.lb2[3]) : uint32_t(P.start_state);

    // --------------------------------------------------------------- S6b
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
        constexpr int K3 = NS > 0 ? NS : 1;
        uint64_t a[K3], zero[K3], ex[K3];
#pragma unroll
        for (int c = 0; c < K3; ++c) {
          a[c] = (tot[c >> 2] >> (16 * (c & 3))) & 0xFFFFull;
          zero[c] = 0;
        }
        lookback_vec<K3>(P.s.lb3_flag, P.s.lb3_agg, P.s.lb3_inc, tile, a, zero, zero,
                         AddOp<K3>{}, cfg, ex);
        if (lane == 0) {
          uint32_t R = 0;
#pragma unroll
          for (int c = 0; c < K3; ++c) {
            if (c < P.n_str) {
              S.base[c] = ex[c];
              S.total[c] = uint32_t(a[c]);
              const uintptr_t g = reinterpret_cast<uintptr_t>(P.chars[c]) + ex[c];
              R = ((R + 15u) & ~15u) + uint32_t(g & 15u);
              S.R[c] = R;
              R += uint32_t(a[c]);
              if (last_tile) P.st->chars_len[P.strcol[c]] = ex[c] + a[c];
            }
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < NSW; ++k) cex[k] = S.wcnt[warp][k] + (ci[k] - cnt[k]);
    }

    // ---------------------------------------------------------------- S7/S8
    const uint32_t rows = S.rows;
    const uint32_t n_out = S.n_out;
    const uint32_t rpb = max(1u, uint32_t(SLOT_CAP) / n_cols);  // rows per pass
    uint64_t rec_end = rec0;
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
            if (lo == 0) {  // stage this chunk's value bytes once
              uint32_t dst = S.R[si] + get16(cex, si) + get16(loc, si);
              for (uint32_t m = seg; m; m &= m - 1) {
                const uint32_t jj = __ffs(m) - 1;
                stage_s[dst++] = own[(jj >> 2) * (4 * NT) + (jj & 3)];
              }
            }
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
      // one lane per field, column-major: a warp handles one column (type)
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
          uint64_t val = 0;
          int err = 0;
          uint64_t fs = 0;
          if (v != SLOT_DEFAULT) {
            const uint32_t fsr = v >> 16;
            const uint64_t fe = tile_base + (v & 0xFFFFu);
            fs = fsr == 0xFFFFu ? tile_fstart : tile_base + fsr;
            if (ty == PP_COL_FLOAT64) {
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
      }
      __syncthreads();
    }
    if (owns_end) P.st->n_records = rec_end;

    // ------------------------------------------- S7b: staged chars -> HBM
    if (NS > 0 && P.has_out) {
      for (int c = 0; c < P.n_str; ++c) {
        uint32_t len = S.total[c];
        if (!len) continue;
        const uint64_t gb = S.base[c];
        if (gb + len > P.chars_cap[c]) {
          if (t == 0) report(P.st, PP_ERR_CAPACITY, 0, false);
          len = gb >= P.chars_cap[c] ? 0u : uint32_t(P.chars_cap[c] - gb);
        }
        uint8_t* g = P.chars[c] + gb;
        const uint8_t* sp = stage_s + S.R[c];
        const uint32_t head = min(len, uint32_t((16u - (reinterpret_cast<uintptr_t>(g) & 15u)) & 15u));
        const uint32_t nvec = (len - head) >> 4;
        const uint32_t tail0 = head + (nvec << 4);
        if (uint32_t(t) < head) g[t] = sp[t];
        uint4* gv = reinterpret_cast<uint4*>(g + head);
        const uint4* sv = reinterpret_cast<const uint4*>(sp + head);
        for (uint32_t v = t; v < nvec; v += NT) __stcs(gv + v, sv[v]);
        if (tail0 + t < len) g[tail0 + t] = sp[tail0 + t];
      }
    }
    if (t == 0) S.tile = S.next_tile;
    __syncthreads();
  }
  // never leave with a bulk copy in flight into this CTA's shared memory
  if (t == 0 && S.issued) mbar_wait_bounded(&S.bar, S.parity, WAIT_LIMIT);
}

// Zero the look-back flags and the tile counter; initialise the status and
// offsets[c][0] = 0 for every string column.
__global__ void parse_init_kernel(uint4* flags, size_t n16, pp_status* st, ParseParams P) {
  const size_t i0 = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < n16; i += size_t(gridDim.x) * blockDim.x) flags[i] = make_uint4(0, 0, 0, 0);
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

template <int NS>
cudaError_t launch_ns(const ParseParams& p, cudaStream_t stream) {
  static int blocks_per_sm = -1, n_sm = 0;
  cudaError_t e;
  if (blocks_per_sm < 0) {
    int dev;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(parse_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(SMEM_BYTES))) != cudaSuccess)
      return e;
    int b = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, parse_kernel<NS>, NT, SMEM_BYTES)) !=
        cudaSuccess)
      return e;
    blocks_per_sm = b > 0 ? b : 1;
  }
  const uint32_t grid = uint32_t(std::min<uint64_t>(p.n_tiles, uint64_t(n_sm) * blocks_per_sm));
  parse_kernel<NS><<<grid, NT, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace ppi {

size_t parse_tile_bytes() { return TILE; }

int parse_ns_width(int n_str) {
  if (n_str <= 0) return 0;
  if (n_str <= 4) return 4;
  if (n_str <= 8) return 8;
  return 16;
}

// layout: [counter 16 B][lb1 8n][lb2_flag 4n][lb3_flag 4n] (zeroed region,
// padded to 16 B) then lb2_agg, lb2_inc (32n each), lb3_agg, lb3_inc (8*ns*n)
static size_t zero_region(uint32_t n) { return (16 + size_t(n) * 16 + 15) & ~size_t(15); }

size_t parse_scratch_bytes(uint32_t n, int ns) {
  const int k3 = ns > 0 ? ns : 1;
  return align256(zero_region(n)) + 2 * align256(size_t(n) * 32) + 2 * align256(size_t(n) * 8 * k3);
}

void parse_scratch_carve(void* base, uint32_t n, int ns, ParseScratch* o) {
  const int k3 = ns > 0 ? ns : 1;
  uint8_t* p = static_cast<uint8_t*>(base);
  o->tile_counter = reinterpret_cast<uint32_t*>(p);
  o->lb1 = reinterpret_cast<unsigned long long*>(p + 16);
  o->lb2_flag = reinterpret_cast<uint32_t*>(p + 16 + size_t(n) * 8);
  o->lb3_flag = reinterpret_cast<uint32_t*>(p + 16 + size_t(n) * 12);
  p += align256(zero_region(n));
  o->lb2_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 32);
  o->lb2_inc = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 32);
  o->lb3_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 8 * k3);
  o->lb3_inc = reinterpret_cast<uint64_t*>(p);
}

cudaError_t launch_parse_init(const ParseParams& p, size_t, void* scratch, cudaStream_t stream) {
  const size_t n16 = zero_region(p.n_tiles) / 16;
  const int threads = 256;
  const int blocks = int(std::min<size_t>((n16 + threads - 1) / threads + 1, 1024));
  parse_init_kernel<<<blocks, threads, 0, stream>>>(static_cast<uint4*>(scratch), n16, p.st, p);
  return cudaGetLastError();
}

cudaError_t launch_parse(const ParseParams& p, cudaStream_t stream) {
  if (p.n_tiles == 0) return cudaSuccess;
  switch (parse_ns_width(p.n_str)) {
    case 0: return launch_ns<0>(p, stream);
    case 4: return launch_ns<4>(p, stream);
    case 8: return launch_ns<8>(p, stream);
    default: return launch_ns<16>(p, stream);
  }
}

}  // namespace ppi
