// General-DFA kernels (|S| <= 16) on sm_103a: pp_tags (per-byte state and
// tag, the test hook) and pp_tokenize (token triples).
//
// The state-transition vector of a chunk (ParPaRaw Section 3.1, Figure 2)
// holds 16 lanes as bytes in four registers.  Each input byte composes it
// with the byte's symbol-group transition (G := G o delta_g, processing the
// chunk back to front): every output word takes two byte-permutes (states
// 0-7 and 8-15) and one bitwise select.  Vectors are composed across the
// warp by shuffles, across the block through shared memory, and across
// tiles by a single-pass decoupled look-back (the exclusive composite scan
// of ParPaRaw Section 3.1).  Each thread then re-runs one DFA from its true
// start state over its chunk.
//
// Tokens (prefix-scan lexing as in "Lexing on the GPU: the scan is the easy
// part", section "A lexer is a prefix scan"): a token starts at byte 0 and
// at every byte tagged PP_TAG_BEGIN; token starts are counted per chunk and
// scanned (second look-back, which also carries the position of the last
// token start) so each start knows its token index; the start of token k
// closes token k-1 (its length and, from the state before the start, its
// id).  The token pass steps the DFA through a per-group row held in
// registers, and a tile's triples are staged in shared memory and written
// with coalesced stores (tiles with more than TOK_CAP tokens write directly).
#include <cstdint>
#include <cuda_runtime.h>
#include <algorithm>

#include "pp.h"
#include "pp_device.cuh"
#include "pp_internal.h"

namespace {
using namespace ppd;
using ppi::GenericDfa;

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int CB = 32;
constexpr int TILE = NT * CB;

// Per symbol group, for the 16-lane composition G' = G o delta_g:
//   sel[k]  PRMT selector for output word k (nibble j = delta_g[4k+j] & 7)
//   msk[k]  0xFF in byte j where delta_g[4k+j] >= 8 (take the high pool)
struct GroupOps {
  uint32_t sel01, sel23;
  uint32_t msk[4];
  uint32_t pad[2];
};

struct Stv16 { uint32_t w[4]; };

__device__ __forceinline__ Stv16 stv16_id() {
  return {{0x03020100u, 0x07060504u, 0x0B0A0908u, 0x0F0E0D0Cu}};
}
__device__ __forceinline__ uint32_t pick(const Stv16& g, uint32_t sel, uint32_t m) {
  const uint32_t lo = __byte_perm(g.w[0], g.w[1], sel);
  const uint32_t hi = __byte_perm(g.w[2], g.w[3], sel);
  return (lo & ~m) | (hi & m);
}
// G o delta_g
__device__ __forceinline__ Stv16 stv16_step(const Stv16& g, const GroupOps& o) {
  Stv16 r;
  r.w[0] = pick(g, o.sel01, o.msk[0]);
  r.w[1] = pick(g, o.sel01 >> 16, o.msk[1]);
  r.w[2] = pick(g, o.sel23, o.msk[2]);
  r.w[3] = pick(g, o.sel23 >> 16, o.msk[3]);
  return r;
}
// (a o b)[i] = b[a[i]]  (a = earlier)
__device__ __forceinline__ Stv16 stv16_compose(const Stv16& a, const Stv16& b) {
  Stv16 r;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t v = a.w[k] & 0x07070707u;
    const uint32_t x = v | (v >> 4);
    const uint32_t sel = __byte_perm(x, 0, 0x0020);
    const uint32_t m = ((a.w[k] >> 3) & 0x01010101u) * 0xFFu;
    r.w[k] = pick(b, sel, m);
  }
  return r;
}
__device__ __forceinline__ uint32_t stv16_apply(const Stv16& g, uint32_t s) {
  const uint32_t k = s >> 2;
  const uint32_t w = k == 0 ? g.w[0] : k == 1 ? g.w[1] : k == 2 ? g.w[2] : g.w[3];
  return (w >> (8 * (s & 3))) & 0xFFu;
}
__device__ __forceinline__ Stv16 shfl_up16(const Stv16& g, int d) {
  return {{__shfl_up_sync(FULL, g.w[0], d), __shfl_up_sync(FULL, g.w[1], d),
           __shfl_up_sync(FULL, g.w[2], d), __shfl_up_sync(FULL, g.w[3], d)}};
}

struct ComposeOp {
  __device__ void operator()(const uint64_t (&a)[2], const uint64_t (&b)[2], uint64_t (&o)[2]) const {
    const Stv16 A = {{uint32_t(a[0]), uint32_t(a[0] >> 32), uint32_t(a[1]), uint32_t(a[1] >> 32)}};
    const Stv16 B = {{uint32_t(b[0]), uint32_t(b[0] >> 32), uint32_t(b[1]), uint32_t(b[1] >> 32)}};
    const Stv16 R = stv16_compose(A, B);
    o[0] = uint64_t(R.w[0]) | (uint64_t(R.w[1]) << 32);
    o[1] = uint64_t(R.w[2]) | (uint64_t(R.w[3]) << 32);
  }
};

struct SharedG {
  uint32_t tile;
  uint32_t pad;
  uint64_t pre[2];
  Stv16 warp_stv[NW];
  uint64_t lb2[2];
  uint32_t tile_cnt;
  uint32_t warp_cnt[NW];
  uint32_t warp_last[NW];
  GroupOps ops[PP_MAX_GROUPS];
  uint8_t grp[256];
  uint8_t delta[PP_MAX_GROUPS * PP_MAX_STATES];  // [group][state]
  uint8_t tag[PP_MAX_STATES * PP_MAX_GROUPS];    // [state][group]
  uint8_t token_id[PP_MAX_STATES];
  uint8_t byte_token_id[256];
};

struct GParams {
  const uint8_t* in;
  uint64_t n;
  uint32_t n_tiles;
  uint32_t spin_limit;
  GenericDfa dfa;
  // tags
  uint8_t* state_before;
  uint8_t* tag;
  // tokens
  uint8_t* out_id;
  uint64_t* out_start;
  uint32_t* out_len;
  uint64_t cap;
  pp_status* st;
  uint32_t* tile_counter;
  uint32_t* lb1_flag;
  uint64_t* lb1_agg;
  uint64_t* lb1_inc;
  uint32_t* lb2_flag;
  uint64_t* lb2_agg;
  uint64_t* lb2_inc;
};

__device__ void setup_tables(const GParams& P, SharedG& S) {
  const int t = threadIdx.x;
  for (int k = t; k < 256; k += NT) {
    S.grp[k] = P.dfa.byte_to_group[k];
    S.byte_token_id[k] = P.dfa.byte_token_id[k];
  }
  for (int k = t; k < PP_MAX_GROUPS * PP_MAX_STATES; k += NT) {
    S.delta[k] = (&P.dfa.delta[0][0])[k];
    S.tag[k] = (&P.dfa.tag[0][0])[k];
  }
  if (t < PP_MAX_STATES) S.token_id[t] = P.dfa.token_id[t];
  if (t < PP_MAX_GROUPS) {
    GroupOps o;
    uint32_t sel[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      o.msk[k] = 0;
      for (int j = 0; j < 4; ++j) {
        const uint32_t d = P.dfa.delta[t][4 * k + j] & 0xFu;
        sel[k] |= (d & 7u) << (4 * j);
        if (d >= 8) o.msk[k] |= 0xFFu << (8 * j);
      }
    }
    o.sel01 = sel[0] | (sel[1] << 16);
    o.sel23 = sel[2] | (sel[3] << 16);
    o.pad[0] = o.pad[1] = 0;
    S.ops[t] = o;
  }
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

// Chunk STV + block composition + tile look-back; returns the thread's
// start state.
__device__ uint32_t resolve_start_state(const GParams& P, SharedG& S, const uint8_t* tile_s,
                                        uint32_t tile, uint32_t cstart, uint32_t clen,
                                        const LookbackCfg& cfg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Stv16 G = stv16_id();
  if (clen == CB) {  // full chunk: unrolled, so every load is issued ahead of the chain
    const uint4* src = reinterpret_cast<const uint4*>(tile_s + cstart);
    const uint4 a = src[0], b = src[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = CB - 1; j >= 0; --j)
      G = stv16_step(G, S.ops[S.grp[(w[j >> 2] >> (8 * (j & 3))) & 0xFFu]]);
  } else {
    for (int j = int(clen) - 1; j >= 0; --j) G = stv16_step(G, S.ops[S.grp[tile_s[cstart + j]]]);
  }
  Stv16 inc = G;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Stv16 o = shfl_up16(inc, d);
    if (lane >= d) inc = stv16_compose(o, inc);
  }
  Stv16 lex = shfl_up16(inc, 1);
  if (lane == 0) lex = stv16_id();
  if (lane == 31) S.warp_stv[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Stv16 wi = lane < NW ? S.warp_stv[lane] : stv16_id();
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
      const Stv16 o = shfl_up16(wi, d);
      if (lane >= d) wi = stv16_compose(o, wi);
    }
    Stv16 wex = shfl_up16(wi, 1);
    if (lane == 0) wex = stv16_id();
    Stv16 agg;
#pragma unroll
    for (int k = 0; k < 4; ++k) agg.w[k] = __shfl_sync(FULL, wi.w[k], NW - 1);
    if (lane < NW) S.warp_stv[lane] = wex;
    const Stv16 id = stv16_id();
    const uint64_t a2[2] = {uint64_t(agg.w[0]) | (uint64_t(agg.w[1]) << 32),
                            uint64_t(agg.w[2]) | (uint64_t(agg.w[3]) << 32)};
    const uint64_t i2[2] = {uint64_t(id.w[0]) | (uint64_t(id.w[1]) << 32),
                            uint64_t(id.w[2]) | (uint64_t(id.w[3]) << 32)};
    uint64_t ex[2];
    lookback_vec<2>(P.lb1_flag, P.lb1_agg, P.lb1_inc, tile, a2, i2, i2, ComposeOp{}, cfg, ex);
    if (lane == 0) { S.pre[0] = ex[0]; S.pre[1] = ex[1]; }
  }
  __syncthreads();
  const Stv16 pre = {{uint32_t(S.pre[0]), uint32_t(S.pre[0] >> 32), uint32_t(S.pre[1]),
                      uint32_t(S.pre[1] >> 32)}};
  uint32_t s = stv16_apply(pre, P.dfa.start_state);
  s = stv16_apply(S.warp_stv[warp], s);
  return stv16_apply(lex, s);
}

__global__ void __launch_bounds__(NT, 2) tags_kernel(const __grid_constant__ GParams P) {
  extern __shared__ __align__(16) uint8_t dyn[];
  uint8_t* tile_s = dyn;
  uint8_t* sb_s = dyn + TILE;
  uint8_t* tg_s = dyn + 2 * TILE;
  __shared__ SharedG S;
  const int t = threadIdx.x;
  setup_tables(P, S);
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t inv = P.dfa.invalid_state;
  for (;;) {
    __syncthreads();
    if (t == 0) S.tile = atomicAdd(P.tile_counter, 1u);
    __syncthreads();
    const uint32_t tile = S.tile;
    if (tile >= P.n_tiles) break;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    load_tile(P.in + tile_base, tile_len, tile_s, t);
    __syncthreads();
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    uint32_t s = resolve_start_state(P, S, tile_s, tile, cstart, clen, cfg);
    for (uint32_t j = 0; j < clen; ++j) {
      const uint32_t g = S.grp[tile_s[cstart + j]];
      const uint32_t nx = S.delta[g * PP_MAX_STATES + s];
      sb_s[cstart + j] = uint8_t(s);
      tg_s[cstart + j] = S.tag[s * PP_MAX_GROUPS + g];
      if (nx == inv && s != inv) report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + j, true);
      s = nx;
    }
    if (tile + 1 == P.n_tiles && clen > 0 && cstart + clen == tile_len && s != inv &&
        !((P.dfa.accept_mask >> s) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    __syncthreads();
    for (uint32_t k = t; k < tile_len; k += NT) {
      P.state_before[tile_base + k] = sb_s[k];
      P.tag[tile_base + k] = tg_s[k];
    }
  }
}

// Per symbol group, the whole transition row for the token pass: next
// state of every state (4-bit lanes, states 0-7 in lo, 8-15 in hi), the
// states in which the group begins a token, and those in which it leads
// into the invalid state.  The state chain then needs no memory access.
struct TokRow { uint32_t lo, hi, begin, to_inv; };

constexpr uint32_t TOK_CAP = 4096;  // tokens per tile staged for coalesced stores

__device__ __forceinline__ uint32_t row_next(const TokRow& r, uint32_t s) {
  return ((s < 8 ? r.lo : r.hi) >> (4 * (s & 7))) & 0xFu;
}

// id of a token from the state after its last byte (or, for 0xFE, from its
// first byte)
__device__ __forceinline__ uint32_t token_id_of(const GParams& P, const SharedG& S,
                                                const uint8_t* tile_s, uint64_t tile_base,
                                                uint32_t s_after, uint64_t start) {
  uint32_t id = S.token_id[s_after];
  if (id == 0xFEu) {
    const uint32_t fb = start >= tile_base ? tile_s[start - tile_base] : __ldg(P.in + start);
    id = S.byte_token_id[fb];
  }
  return id;
}

__global__ void __launch_bounds__(NT, 2) tokenize_kernel(const __grid_constant__ GParams P) {
  extern __shared__ __align__(16) uint8_t dyn[];
  uint8_t* tile_s = dyn;                                            // TILE
  uint8_t* sc_s = dyn + TILE;                                       // [32][NT]: state before each start
  uint16_t* start_s = reinterpret_cast<uint16_t*>(dyn + 2 * TILE);  // [TOK_CAP]
  uint32_t* len_s = reinterpret_cast<uint32_t*>(start_s + TOK_CAP); // [TOK_CAP + 1]
  uint8_t* id_s = reinterpret_cast<uint8_t*>(len_s + TOK_CAP + 1);  // [TOK_CAP + 1]
  __shared__ SharedG S;
  __shared__ TokRow rows[PP_MAX_GROUPS];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  setup_tables(P, S);
  if (t < PP_MAX_GROUPS) {
    TokRow r = {0u, 0u, 0u, 0u};
    for (uint32_t st = 0; st < uint32_t(P.dfa.n_states); ++st) {
      const uint32_t nx = P.dfa.delta[t][st] & 0xFu;
      if (st < 8) r.lo |= nx << (4 * st);
      else r.hi |= nx << (4 * (st - 8));
      if (P.dfa.tag[st][t] == PP_TAG_BEGIN) r.begin |= 1u << st;
      if (nx == P.dfa.invalid_state && st != P.dfa.invalid_state) r.to_inv |= 1u << st;
    }
    rows[t] = r;
  }
  const LookbackCfg cfg{P.st, P.spin_limit};
  const uint32_t inv = P.dfa.invalid_state;
  for (;;) {
    __syncthreads();
    if (t == 0) S.tile = atomicAdd(P.tile_counter, 1u);
    __syncthreads();
    const uint32_t tile = S.tile;
    if (tile >= P.n_tiles) break;
    const uint64_t tile_base = uint64_t(tile) * TILE;
    const uint32_t tile_len = uint32_t(min(uint64_t(TILE), P.n - tile_base));
    const bool last_tile = tile + 1 == P.n_tiles;
    load_tile(P.in + tile_base, tile_len, tile_s, t);
    __syncthreads();
    const uint32_t cstart = uint32_t(t) * CB;
    const uint32_t clen = tile_len > cstart ? min(tile_len - cstart, uint32_t(CB)) : 0u;
    const uint32_t s0 = resolve_start_state(P, S, tile_s, tile, cstart, clen, cfg);

    // token starts of the chunk; the state before each is kept for its id
    uint32_t begin = 0, s = s0, last_start = 0, nb = 0, inv_at = 32;
    auto step = [&](uint32_t j, uint32_t byte) {
      const TokRow r = rows[S.grp[byte]];
      if (((r.begin >> s) & 1u) || (tile_base + cstart + j == 0)) {
        begin |= 1u << j;
        sc_s[nb * NT + t] = uint8_t(s);
        ++nb;
      }
      if (((r.to_inv >> s) & 1u) && inv_at == 32) inv_at = j;
      s = row_next(r, s);
    };
    if (clen == CB) {  // full chunk: unrolled, loads ahead of the state chain
      const uint4* src = reinterpret_cast<const uint4*>(tile_s + cstart);
      const uint4 a = src[0], b = src[1];
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (uint32_t j = 0; j < CB; ++j) step(j, (w[j >> 2] >> (8 * (j & 3))) & 0xFFu);
    } else {
      for (uint32_t j = 0; j < clen; ++j) step(j, tile_s[cstart + j]);
    }
    if (begin) last_start = cstart + (31u - __clz(begin)) + 1u;
    if (inv_at < 32) report(P.st, PP_ERR_INVALID_INPUT, tile_base + cstart + inv_at, true);
    const uint32_t s_end = s;
    const bool owns_end = last_tile && clen > 0 && cstart + clen == tile_len;
    if (owns_end && s_end != inv && !((P.dfa.accept_mask >> s_end) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);

    // token index scan: (count, last start pos+1)
    uint32_t ci = nb, li = last_start;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t oc = __shfl_up_sync(FULL, ci, d), ol = __shfl_up_sync(FULL, li, d);
      if (lane >= d) { ci += oc; li = li ? li : ol; }
    }
    uint32_t lc = __shfl_up_sync(FULL, ci, 1), ll = __shfl_up_sync(FULL, li, 1);
    if (lane == 0) { lc = 0; ll = 0; }
    if (lane == 31) { S.warp_cnt[warp] = ci; S.warp_last[warp] = li; }
    __syncthreads();
    if (warp == 0) {
      const uint32_t vc = lane < NW ? S.warp_cnt[lane] : 0u;
      const uint32_t vl = lane < NW ? S.warp_last[lane] : 0u;
      uint32_t wc = vc, wl = vl;
#pragma unroll
      for (int d = 1; d < NW; d <<= 1) {
        const uint32_t oc = __shfl_up_sync(FULL, wc, d), ol = __shfl_up_sync(FULL, wl, d);
        if (lane >= d) { wc += oc; wl = wl ? wl : ol; }
      }
      const uint32_t tc = __shfl_sync(FULL, wc, NW - 1), tl = __shfl_sync(FULL, wl, NW - 1);
      if (lane < NW) { S.warp_cnt[lane] = wc - vc; }
      uint32_t ex_l = __shfl_up_sync(FULL, wl, 1);
      if (lane == 0) ex_l = 0;
      if (lane < NW) S.warp_last[lane] = ex_l;
      if (lane == 0) S.tile_cnt = tc;
      const uint64_t a2[2] = {tc, tl ? tile_base + tl : 0ull};
      const uint64_t z[2] = {0ull, 0ull};
      uint64_t ex[2];
      lookback_vec<2>(P.lb2_flag, P.lb2_agg, P.lb2_inc, tile, a2, z, z,
                      [](const uint64_t (&a)[2], const uint64_t (&b)[2], uint64_t (&o)[2]) {
                        o[0] = a[0] + b[0];
                        o[1] = b[1] ? b[1] : a[1];
                      },
                      cfg, ex);
      if (lane == 0) { S.lb2[0] = ex[0]; S.lb2[1] = ex[1]; }
    }
    __syncthreads();
    const uint64_t k0 = S.lb2[0];                 // first token starting in this tile
    const uint32_t c = S.tile_cnt;                // tokens starting in this tile
    const uint32_t i0 = S.warp_cnt[warp] + lc;    // this chunk's first start, tile-local
    uint64_t prev_start1;                         // start (+1) of the token open at the chunk start
    if (ll) prev_start1 = tile_base + ll;
    else if (S.warp_last[warp]) prev_start1 = tile_base + S.warp_last[warp];
    else prev_start1 = S.lb2[1];
    const bool staged = c <= TOK_CAP;
    const bool sizing = P.cap == 0 && P.out_start == nullptr;

    // emit: each start opens token k0 + i and closes token k0 + i - 1
    {
      uint32_t m = begin, b = 0;
      while (m) {
        const uint32_t j = __ffs(m) - 1;
        m &= m - 1;
        const uint32_t i = i0 + b;
        const uint64_t pos = tile_base + cstart + j;
        const uint32_t sb = sc_s[b * NT + t];
        ++b;
        uint32_t id = 0, len = 0;
        const bool closes = prev_start1 != 0;
        if (closes) {
          const uint64_t ps = prev_start1 - 1;
          id = token_id_of(P, S, tile_s, tile_base, sb, ps);
          len = uint32_t(pos - ps);
        }
        if (staged) {
          start_s[i] = uint16_t(cstart + j);
          len_s[i] = len;
          id_s[i] = uint8_t(id);
        } else {
          const uint64_t k = k0 + i;
          if (closes && k - 1 < P.cap) { P.out_id[k - 1] = uint8_t(id); P.out_len[k - 1] = len; }
          if (k < P.cap) P.out_start[k] = pos;
          else if (!sizing) report(P.st, PP_ERR_CAPACITY, 0, false);
        }
        prev_start1 = pos + 1;
      }
      if (owns_end) {  // close the last token
        const uint64_t k = k0 + i0 + b;  // tokens in total
        if (prev_start1) {
          const uint64_t ps = prev_start1 - 1;
          const uint32_t id = token_id_of(P, S, tile_s, tile_base, s_end, ps);
          const uint32_t len = uint32_t(P.n - ps);
          if (staged) { len_s[c] = len; id_s[c] = uint8_t(id); }
          else if (k - 1 < P.cap) { P.out_id[k - 1] = uint8_t(id); P.out_len[k - 1] = len; }
        }
        P.st->n_tokens = k;
      }
    }
    if (staged) {
      __syncthreads();
      // starts of tokens k0 .. k0+c-1; ids and lengths of tokens k0-1 .. k0+c-2
      // (and k0+c-1 in the last tile)
      const uint32_t nclose = c + (last_tile ? 1u : 0u);
      for (uint32_t i = t; i < nclose; i += NT) {
        const uint64_t k = k0 + i;
        if (i < c) {
          if (k < P.cap) P.out_start[k] = tile_base + start_s[i];
          else if (!sizing) report(P.st, PP_ERR_CAPACITY, 0, false);
        }
        if (k >= 1 && k - 1 < P.cap) {  // token k-1 exists (the first start closes none)
          P.out_len[k - 1] = len_s[i];
          P.out_id[k - 1] = id_s[i];
        }
      }
    }
  }
}

__global__ void generic_init_kernel(uint4* zero, size_t n16, pp_status* st) {
  const size_t i0 = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < n16; i += size_t(gridDim.x) * blockDim.x) zero[i] = make_uint4(0, 0, 0, 0);
  if (i0 == 0) {
    st->error = 0;
    st->reserved = 0;
    st->first_error_offset = ~0ull;
    st->n_records = 0;
    st->n_tokens = 0;
    for (int c = 0; c < PP_MAX_COLS; ++c) st->chars_len[c] = 0;
  }
}

__global__ void count_byte_kernel(const uint8_t* in, uint64_t n, uint8_t value, uint64_t* out) {
  uint64_t c = 0;
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  const uint64_t i0 = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(in) & 15) == 0) {
    const uint64_t nv = n >> 4;
    const uint4* v = reinterpret_cast<const uint4*>(in);
    const uint32_t rep = 0x01010101u * value;
    for (uint64_t i = i0; i < nv; i += stride) {
      const uint4 x = __ldcs(v + i);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t z = w[q] ^ rep;  // zero bytes where equal
        const uint32_t hi = ~(((z & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | z | 0x7F7F7F7Fu);
        c += __popc(hi);
      }
    }
    for (uint64_t i = (nv << 4) + i0; i < n; i += stride) c += in[i] == value;
  } else {
    for (uint64_t i = i0; i < n; i += stride) c += in[i] == value;
  }
  for (int d = 16; d; d >>= 1) c += __shfl_down_sync(FULL, c, d);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(reinterpret_cast<unsigned long long*>(out), c);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// [counter 16][lb1_flag 4n][lb2_flag 4n] zeroed, then lb1_agg/inc, lb2_agg/inc (16n each)
size_t zero_bytes(uint32_t n) { return (16 + size_t(n) * 8 + 15) & ~size_t(15); }

void carve(void* base, uint32_t n, GParams& P) {
  uint8_t* p = static_cast<uint8_t*>(base);
  P.tile_counter = reinterpret_cast<uint32_t*>(p);
  P.lb1_flag = reinterpret_cast<uint32_t*>(p + 16);
  P.lb2_flag = reinterpret_cast<uint32_t*>(p + 16 + size_t(n) * 4);
  p += align256(zero_bytes(n));
  P.lb1_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 16);
  P.lb1_inc = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 16);
  P.lb2_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 16);
  P.lb2_inc = reinterpret_cast<uint64_t*>(p);
}

uint32_t n_tiles_of(uint64_t n) { return uint32_t((n + TILE - 1) / TILE); }

cudaError_t run(void (*kern)(GParams), size_t dyn_smem, const GParams& P, void* scratch,
                cudaStream_t stream) {
  const size_t n16 = zero_bytes(P.n_tiles) / 16;
  generic_init_kernel<<<int(std::min<size_t>((n16 + 255) / 256 + 1, 1024)), 256, 0, stream>>>(
      static_cast<uint4*>(scratch), n16, P.st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || P.n_tiles == 0) return e;
  static int n_sm = 0;
  if (!n_sm) {
    int dev;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
  }
  if (dyn_smem > 0 &&
      (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn_smem))) !=
          cudaSuccess)
    return e;
  const uint32_t grid = std::min<uint32_t>(P.n_tiles, uint32_t(n_sm) * 2);
  kern<<<grid, NT, dyn_smem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace

namespace ppi {

extern uint32_t g_spin_limit;

size_t tags_scratch_bytes(uint64_t n) {
  const uint32_t nt = n_tiles_of(n);
  return align256(zero_bytes(nt)) + 4 * align256(size_t(nt) * 16);
}
size_t tokenize_scratch_bytes(uint64_t n) { return tags_scratch_bytes(n); }

cudaError_t launch_tags(const uint8_t* in, uint64_t n, const GenericDfa& dfa,
                        uint8_t* state_before, uint8_t* tag, pp_status* st, void* scratch,
                        size_t, cudaStream_t stream) {
  GParams P{};
  P.in = in;
  P.n = n;
  P.n_tiles = n_tiles_of(n);
  P.spin_limit = g_spin_limit;
  P.dfa = dfa;
  P.state_before = state_before;
  P.tag = tag;
  P.st = st;
  carve(scratch, P.n_tiles, P);
  return run(tags_kernel, 3 * TILE, P, scratch, stream);
}

cudaError_t launch_tokenize(const uint8_t* in, uint64_t n, const GenericDfa& dfa,
                            uint8_t* out_id, uint64_t* out_start, uint32_t* out_len,
                            uint64_t cap, pp_status* st, void* scratch, size_t,
                            cudaStream_t stream) {
  GParams P{};
  P.in = in;
  P.n = n;
  P.n_tiles = n_tiles_of(n);
  P.spin_limit = g_spin_limit;
  P.dfa = dfa;
  P.out_id = out_id;
  P.out_start = out_start;
  P.out_len = out_len;
  P.cap = cap;
  P.st = st;
  carve(scratch, P.n_tiles, P);
  return run(tokenize_kernel, 2 * TILE + TOK_CAP * 2 + (TOK_CAP + 1) * 5, P, scratch, stream);
}

cudaError_t launch_count_byte(const uint8_t* in, uint64_t n, uint8_t value, uint64_t* d_count,
                              cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(d_count, 0, sizeof(uint64_t), stream);
  if (e != cudaSuccess || n == 0) return e;
  static int n_sm = 0;
  if (!n_sm) {
    int dev;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
  }
  const uint64_t want = (n / 16 + 255) / 256;
  const int blocks = int(std::min<uint64_t>(want ? want : 1, uint64_t(n_sm) * 8));
  count_byte_kernel<<<blocks, 256, 0, stream>>>(in, n, value, d_count);
  return cudaGetLastError();
}

}  // namespace ppi
