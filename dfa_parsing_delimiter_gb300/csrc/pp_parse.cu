// pp_parse: single-pass DFA-based parsing of delimiter-separated input into
// Arrow-style columns on sm_103a.
//
// One persistent CTA of 512 threads works on 16 KiB tiles taken in order
// from an atomic counter.  Per tile:
//   S1  the tile is loaded into shared memory once (16-byte coalesced loads);
//       HBM input is read exactly once.
//   S2  each thread runs the multi-instance DFA over its 32-byte chunk
//       (ParPaRaw Section 3.1, Figure 2): the state-transition vector of all
//       live states sits in one register, one byte per state, and each input
//       byte composes it with the byte's symbol-group transition by one
//       byte-permute (PRMT) — the row-per-symbol-group transition table of
//       ParPaRaw Section 5 (Table 1), fetched from a per-lane replicated
//       shared-memory LUT so the lookup never bank-conflicts.
//   S3  warp shuffles and a block pass compose the vectors; a single-pass
//       decoupled look-back over tiles gives the tile's exclusive composite
//       prefix, seeded with the identity (ParPaRaw Section 3.1).
//   S5  each thread re-runs ONE DFA from its true start state over the
//       chunk's non-background bytes only and builds the three bitmap
//       indexes (record delimiter, field delimiter, control; ParPaRaw
//       Section 3.1).
//   S6  record counts (POPCNT) and absolute/relative column offsets
//       (ParPaRaw Section 3.2, Figure 4) are scanned across the block and the
//       tiles (second look-back), then the per-string-column value-byte
//       counts (third look-back) give each tile its place in every column's
//       chars buffer.
//   S7  value bytes are compacted per column into shared memory and written
//       out as contiguous 16-byte stores (the column-partitioning step of
//       ParPaRaw Section 3.3 as stream compaction instead of a radix sort);
//       Arrow offsets are written by the thread that owns each field's
//       terminator.
//   S8  numeric fields are converted by the terminator's owner (ParPaRaw
//       Section 3.3, thread-exclusive collaboration level).
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
constexpr uint64_t ABS64 = 1ull << 63;
constexpr uint32_t ABS32 = 1u << 31;

struct Shared {
  uint32_t tile;
  uint32_t stv_prefix;
  uint32_t warp_stv[NW];
  uint32_t warp_rec[NW], warp_col[NW], warp_last[NW];
  uint64_t lb2[4];
  uint64_t wcnt[NW][4];
  uint64_t base[ppi::MAX_STR_COLS];
  uint32_t total[ppi::MAX_STR_COLS];
  uint32_t R[ppi::MAX_STR_COLS];
  int8_t stridx[PP_MAX_COLS];
  uint8_t coltype[PP_MAX_COLS];
};

constexpr size_t SMEM_BYTES = LUT_BYTES + TILE + STAGE_BYTES + NT * 4 + sizeof(Shared);

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

__device__ __forceinline__ void load_tile(const uint8_t* g, uint32_t len, uint8_t* s, int t) {
  if ((reinterpret_cast<uintptr_t>(g) & 15) == 0) {
    const uint32_t nv = len >> 4;
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    uint4* sv = reinterpret_cast<uint4*>(s);
    for (uint32_t v = t; v < nv; v += NT) sv[v] = __ldcs(gv + v);
    for (uint32_t k = (nv << 4) + t; k < len; k += NT) s[k] = g[k];
  } else {
    for (uint32_t k = t; k < len; k += NT) s[k] = g[k];
  }
}

// Feed the value bytes of field [fs, fe) (global offsets) to a numeric
// accumulator; returns the number of value bytes.  Fields inside the tile
// use the tile copy and the control bitmap; a field that began in an
// earlier tile is re-read from global memory and re-tagged by running the
// DFA from the state at its first byte.
template <class Acc>
__device__ __forceinline__ uint32_t feed_field(Acc& acc, const uint8_t* in, uint64_t fs,
                                               uint64_t fe, uint64_t tile_base,
                                               const uint8_t* tile_s, const uint32_t* ctrl_s,
                                               const uint32_t* my_lut, uint32_t fstate) {
  uint32_t ndata = 0;
  if (fs >= tile_base) {
    const uint32_t e = uint32_t(fe - tile_base);
    for (uint32_t p = uint32_t(fs - tile_base); p < e; ++p) {
      if ((ctrl_s[p >> 5] >> (p & 31)) & 1u) continue;
      acc.feed(tile_s[p]);
      ++ndata;
    }
  } else {
    uint32_t s = fstate;
    for (uint64_t p = fs; p < fe; ++p) {
      const uint32_t b = p >= tile_base ? uint32_t(tile_s[p - tile_base]) : uint32_t(__ldg(in + p));
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

template <int NS>
__global__ void __launch_bounds__(NT, 2) parse_kernel(const __grid_constant__ ParseParams P) {
  constexpr int NSW = NS > 0 ? (NS + 3) / 4 : 1;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  uint8_t* tile_s = smem + LUT_BYTES;
  uint8_t* stage_s = tile_s + TILE;
  uint32_t* ctrl_s = reinterpret_cast<uint32_t*>(stage_s + STAGE_BYTES);
  Shared& S = *reinterpret_cast<Shared*>(ctrl_s + NT);

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int k = t; k < 256 * 32; k += NT) lut_s[k] = P.lut[k >> 5];
  for (int k = t; k < PP_MAX_COLS; k += NT) {
    S.stridx[k] = P.stridx[k];
    S.coltype[k] = P.coltype[k];
  }
  const uint32_t* my_lut = lut_s + lane;
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t n_cols = uint32_t(P.n_cols);

  for (;;) {
    __syncthreads();
    if (t == 0) S.tile = atomicAdd(P.s.tile_counter, 1u);
    __syncthreads();
    const uint32_t tile = S.tile;
    if (tile >= P.n_tiles) break;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    const bool last_tile = tile + 1 == P.n_tiles;

    // ---------------------------------------------------------------- S1
    load_tile(P.in + tile_base, tile_len, tile_s, t);
    __syncthreads();

    // ---------------------------------------------------------------- S2
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    uint32_t G = STV_ID, special = 0;
    if (clen == CB) {
      const uint4* src = reinterpret_cast<const uint4*>(tile_s + cstart);
      const int sw = (t >> 2) & 1;  // alternate read order: conflict-free 16-byte reads
      const uint4 x = src[sw], y = src[sw ^ 1];
      const uint4 lo = sw ? y : x, hi = sw ? x : y;
      const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int j = CB - 1; j >= 0; --j) {
        const uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        const uint32_t e = my_lut[b << 5];
        G = __byte_perm(G, STV_INV_POOL, e);   // G := G o delta_group(b)
        special = __funnelshift_l(e, special, 1);
      }
    } else {
      for (int j = int(clen) - 1; j >= 0; --j) {
        const uint32_t e = my_lut[uint32_t(tile_s[cstart + j]) << 5];
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
        const uint32_t e = my_lut[uint32_t(tile_s[cstart + j]) << 5];
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
      V2 w = lane < NW ? V2{S.warp_rec[lane], S.warp_col[lane], S.warp_last[lane]} : V2{0u, 0u, 0u};
      V2 wi = w;
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
      if (lane == 0) { S.lb2[0] = ex[0]; S.lb2[1] = ex[1]; S.lb2[2] = ex[2]; S.lb2[3] = ex[3]; }
    }
    __syncthreads();
    const V2 pre = op2_32(V2{S.warp_rec[warp], S.warp_col[warp], S.warp_last[warp]}, lex);
    const uint64_t rec0 = S.lb2[0] + pre.rec;
    uint32_t col0;
    if (pre.col & ABS32) {
      col0 = pre.col & ~ABS32;
    } else {
      const uint64_t c = (S.lb2[1] & ~ABS64) + pre.col;
      col0 = c > 0x7FFFFF00ull ? 0x7FFFFF00u : uint32_t(c);
    }
    uint64_t fstart0;
    uint32_t fstate0;
    if (pre.last) { fstart0 = tile_base + (pre.last >> 8); fstate0 = pre.last & 0xFFu; }
    else if (S.lb2[2]) { fstart0 = S.lb2[2]; fstate0 = uint32_t(S.lb2[3]); }
    else { fstart0 = 0; fstate0 = P.start_state; }

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
          for (int c = 0; c < P.n_str; ++c) {
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
      __syncthreads();
#pragma unroll
      for (int k = 0; k < NSW; ++k) cex[k] = S.wcnt[warp][k] + (ci[k] - cnt[k]);
    }

    // ---------------------------------------------------------------- S7/S8
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
          uint32_t dst = S.R[si] + get16(cex, si) + get16(loc, si);
          for (uint32_t m = seg; m; m &= m - 1) stage_s[dst++] = tile_s[cstart + __ffs(m) - 1];
          add16(loc, si, __popc(seg));
        }
        uint64_t tpos;
        bool is_rd;
        if (j < 32) { tpos = tile_base + cstart + j; is_rd = (rd >> j) & 1u; }
        else if (virt_rd) { tpos = P.n; is_rd = true; }
        else break;
        // close field (col, rec) = bytes [fstart, tpos)
        if (col < n_cols) {
          const uint32_t ty = S.coltype[col];
          if (rec >= P.rec_cap) {
            if (P.has_out && ty != PP_COL_SKIP) report(P.st, PP_ERR_CAPACITY, 0, false);
          } else if (ty == PP_COL_STRING) {
            const uint64_t v = S.base[si] + get16(cex, si) + get16(loc, si);
            if (v > 0x7FFFFFFFull || v > P.chars_cap[si]) {
              if (P.has_out) report(P.st, PP_ERR_CAPACITY, 0, false);
            } else if (P.has_out) {
              P.offsets[si][rec + 1] = int32_t(v);
            }
          } else if (ty == PP_COL_FLOAT64) {
            if (P.has_out) {
              ppn::FloatAcc acc;
              const uint32_t nd = feed_field(acc, P.in, fstart, tpos, tile_base, tile_s, ctrl_s,
                                             my_lut, fstart == fstart0 ? fstate0 : 0u);
              double v = 0.0;
              const int err = nd ? acc.finish(&v) : 0;
              static_cast<double*>(P.typed[col])[rec] = v;
              if (err) report(P.st, err, fstart, true);
            }
          } else if (ty != PP_COL_SKIP) {
            if (P.has_out) {
              ppn::IntAcc acc;
              const uint32_t nd = feed_field(acc, P.in, fstart, tpos, tile_base, tile_s, ctrl_s,
                                             my_lut, fstart == fstart0 ? fstate0 : 0u);
              int64_t v = 0;
              int err = 0;
              if (ty == PP_COL_INT8) {
                if (nd) err = acc.finish(128ull, 127ull, &v);
                static_cast<int8_t*>(P.typed[col])[rec] = int8_t(v);
              } else if (ty == PP_COL_INT32) {
                if (nd) err = acc.finish(2147483648ull, 2147483647ull, &v);
                static_cast<int32_t*>(P.typed[col])[rec] = int32_t(v);
              } else {
                if (nd) err = acc.finish(9223372036854775808ull, 9223372036854775807ull, &v);
                static_cast<int64_t*>(P.typed[col])[rec] = v;
              }
              if (err) report(P.st, err, fstart, true);
            }
          }
        }
        if (is_rd) {
          if (col != n_cols - 1) {
            report(P.st, PP_ERR_COLCOUNT, tpos, true);
            // missing fields take the column default
            for (uint32_t c = col + 1; c < n_cols && rec < P.rec_cap && P.has_out; ++c) {
              const uint32_t ty = S.coltype[c];
              if (ty == PP_COL_STRING) {
                const int sc = S.stridx[c];
                const uint64_t v = S.base[sc] + get16(cex, sc) + get16(loc, sc);
                if (v <= 0x7FFFFFFFull && v <= P.chars_cap[sc]) P.offsets[sc][rec + 1] = int32_t(v);
              } else if (ty == PP_COL_FLOAT64) {
                static_cast<double*>(P.typed[c])[rec] = 0.0;
              } else if (ty == PP_COL_INT8) {
                static_cast<int8_t*>(P.typed[c])[rec] = 0;
              } else if (ty == PP_COL_INT32) {
                static_cast<int32_t*>(P.typed[c])[rec] = 0;
              } else if (ty == PP_COL_INT64) {
                static_cast<int64_t*>(P.typed[c])[rec] = 0;
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
      if (owns_end) P.st->n_records = rec;
    }
    __syncthreads();

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
  }
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
