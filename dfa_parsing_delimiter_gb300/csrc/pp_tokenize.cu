// pp_tokenize on sm_103a: token triples (id, start, length) from a general
// DFA with up to 16 states, in five passes that never wait on one another
// inside a kernel's byte loop.
//
// The input is cut into pieces of 2 KiB, one per warp, 64 bytes per lane.
//   1. stv    Per lane, the state-transition vector of its 64 bytes
//             (ParPaRaw Section 3.1, Figure 2), built back to front three
//             bytes at a time from a table of composed transitions; a
//             warp scan gives each lane the vector of the bytes before it in
//             the piece, and lane 31 the piece's vector.
//   2. scan   Exclusive composite scan of the piece vectors (decoupled
//             look-back over tiles of 4096 pieces); applied to the DFA's
//             start state it gives the state at every piece start.
//   3. count  Each lane re-runs one DFA from its true start state and counts
//             its token starts ("Lexing on the GPU: the scan is the easy
//             part", section "A lexer is a prefix scan": a token starts at
//             byte 0 and wherever a transition is tagged as a token begin).
//   4. scan   Exclusive scan of (token count, position of the last token
//             start) over pieces: the index of every piece's first token and
//             the start of the token open at the piece start.
//   5. emit   The DFA runs again and every token start k writes start[k] and
//             closes token k-1 (its length, and its id from the state before
//             the start).  A piece's triples are staged in shared memory and
//             written with coalesced stores.
// The byte passes read the input straight from HBM with 16-byte loads.  The
// count pass looks up tables replicated per lane in shared memory (no bank
// conflicts); the emit pass steps the DFA two bytes per lookup.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_device.cuh"
#include "pp_internal.h"
#include "pp_stv16.cuh"

namespace {
using namespace ppd;
using ppi::GenericDfa;

constexpr int CB = 64;                   // bytes per lane
constexpr int PIECE = 32 * CB;           // bytes per warp
constexpr int WT = 256;                  // threads per block, transition-vector pass
constexpr int WW = WT / 32;
constexpr int EMIT_BPS = 5;              // emit pass: blocks per SM (48 registers a thread)
constexpr int SCAN_T = 256, SCAN_E = 16; // scan passes: pieces per thread
constexpr int SCAN_TILE = SCAN_T * SCAN_E;
constexpr uint32_t CAPW = 512;           // tokens per piece staged for coalesced stores

struct TokParams {
  const uint8_t* in;
  uint64_t n;
  uint32_t n_pieces;
  uint32_t spin_limit;
  bool aligned;  // in is 16-byte aligned
  GenericDfa dfa;
  uint8_t* out_id;
  uint64_t* out_start;
  uint32_t* out_len;
  uint64_t cap;
  pp_status* st;
  // scratch
  uint32_t* tickets;      // [0] state scan, [1] count scan
  uint32_t* flag_s;       // look-back, state scan
  uint64_t* agg_s;
  uint64_t* inc_s;
  uint32_t* flag_c;       // look-back, count scan
  uint64_t* agg_c;
  uint64_t* inc_c;
  uint64_t* lane_pre;     // [pieces * 32] vector of the piece's bytes before the lane (nibbles)
  uint64_t* piece_stv;    // [pieces] vector of the piece (nibbles)
  uint8_t* piece_state;   // [pieces] state at the piece start
  uint32_t* lane_info;    // [pieces * 32] start state | starts << 4 | (last start + 1) << 11
  uint32_t* piece_cnt;    // [pieces] token starts in the piece
  uint32_t* piece_last;   // [pieces] offset + 1 of the piece's last token start (0: none)
  uint64_t* piece_k0;     // [pieces] index of the piece's first token start
  uint64_t* piece_prev;   // [pieces] start + 1 of the token open at the piece start (0: none)
  // Partial mode (streaming chunks), when not null: the input ends inside
  // its last token, which is left open (no length, id or end-state check);
  // carry_out[0] = 1 + the last token start, carry_out[1] = the DFA state
  // before it.
  unsigned long long* carry_out;
};

// ------------------------------------------------------------ input
// 16 words of r from word WS on, shifted right by sh bits (0, 8, 16, 24).
template <int WS>
__device__ __forceinline__ void shift_words(const uint32_t (&r)[20], uint32_t sh,
                                            uint32_t (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 16; ++q) w[q] = __funnelshift_r(r[WS + q], r[WS + q + 1], sh);
}
// The lane's 64 bytes as 16 little-endian words (zero past clen).  A full
// chunk is read with 16-byte loads: four of them on a 16-byte aligned input;
// otherwise five aligned loads around the chunk, shifted into place, as long
// as they stay inside the input (every chunk but the input's first and
// last).  The misalignment is the same for every chunk (chunks start at
// multiples of 64).
__device__ __forceinline__ void load_chunk(const TokParams& P, uint64_t c0, uint32_t clen,
                                           uint32_t (&w)[16]) {
  const uint32_t m = uint32_t(reinterpret_cast<uintptr_t>(P.in) & 15u);
  if (clen == CB && P.aligned) {
    const uint4* src = reinterpret_cast<const uint4*>(P.in + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(src + q);
      w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
    }
  } else if (clen == CB && c0 >= 16 && c0 + CB + 16 <= P.n) {
    const uint4* src = reinterpret_cast<const uint4*>(P.in + c0 - m);
    uint32_t r[20];
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      const uint4 v = __ldg(src + q);
      r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
    }
    const uint32_t sh = (m & 3u) * 8u;
    switch (m >> 2) {
      case 0: shift_words<0>(r, sh, w); break;
      case 1: shift_words<1>(r, sh, w); break;
      case 2: shift_words<2>(r, sh, w); break;
      default: shift_words<3>(r, sh, w); break;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (uint32_t(4 * q + k) < clen) x |= uint32_t(__ldg(P.in + c0 + 4 * q + k)) << (8 * k);
      w[q] = x;
    }
  }
}
__device__ __forceinline__ uint32_t byte_of(const uint32_t (&w)[16], int j) {
  return (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
}
__device__ __forceinline__ uint32_t chunk_len(uint64_t c0, uint64_t n) {
  return c0 < n ? uint32_t(min(uint64_t(CB), n - c0)) : 0u;
}

// ------------------------------------------------------------ pass 1
// Steps of G'(s) = G(D(s)) take D as selector nibbles: word x holds
// D(0..7) (4 bits each), y D(8..15).  tri[] holds D for three consecutive
// bytes (groups g1, g2, g3: D = delta_g3 o delta_g2 o delta_g1) at entry
// g1 * 256 + g2 * 16 + (g3 ^ g1 ^ rot(g2)), addressed in bytes as
// ga[b1] ^ gb[b2] ^ gc[b3]: the first two groups move the entry's bank, so
// a warp's lanes spread over the banks whatever their third byte.
// single[] holds one byte's D, at gc[b].
struct StvTables {
  uint16_t ga[256];  // group * 2048, and the bank move
  uint16_t gb[256];  // group * 128, and the bank move
  uint16_t gc[256];  // group * 8
  uint2 tri[16 * 16 * 16];
  uint2 single[PP_MAX_GROUPS];
  Stv16 delta[PP_MAX_GROUPS];  // delta_g as a vector (table construction)
};

__device__ __forceinline__ uint32_t tri_rot(uint32_t g) { return ((g >> 2) | (g << 2)) & 15u; }

__device__ __forceinline__ Stv16 stv_step(const Stv16& G, uint2 e) {
  const uint32_t xx = e.x ^ 0x88888888u, xy = e.y ^ 0x88888888u;
  Stv16 r;
  r.w[0] = stv16_gather(G, e.x, xx);
  r.w[1] = stv16_gather(G, e.x >> 16, xx >> 16);
  r.w[2] = stv16_gather(G, e.y, xy);
  r.w[3] = stv16_gather(G, e.y >> 16, xy >> 16);
  return r;
}
__device__ __forceinline__ uint2 as_sel(const Stv16& d) {
  const uint64_t v = stv16_pack(d);
  return make_uint2(uint32_t(v), uint32_t(v >> 32));
}
template <class T>
__device__ __forceinline__ const T& at_byte(const T* base, uint32_t off) {
  return *reinterpret_cast<const T*>(reinterpret_cast<const uint8_t*>(base) + off);
}

__global__ void __launch_bounds__(WT, 4) tok_stv_kernel(const __grid_constant__ TokParams P) {
  __shared__ StvTables S;
  const int t = threadIdx.x, lane = t & 31;
  for (int k = t; k < 256; k += WT) {
    const uint32_t g = P.dfa.byte_to_group[k] & 0xFu;
    S.ga[k] = uint16_t((g << 11) ^ (g << 3));
    S.gb[k] = uint16_t((g << 7) ^ (tri_rot(g) << 3));
    S.gc[k] = uint16_t(g << 3);
  }
  if (t < PP_MAX_GROUPS) {
    Stv16 d;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = 0;
      for (int b = 0; b < 4; ++b) x |= uint32_t(P.dfa.delta[t][4 * k + b] & 0xFu) << (8 * b);
      d.w[k] = x;
    }
    S.delta[t] = d;
    S.single[t] = as_sel(d);
  }
  __syncthreads();
  for (int k = t; k < 16 * 16 * 16; k += WT) {
    const uint32_t g1 = uint32_t(k) >> 8, g2 = (uint32_t(k) >> 4) & 15u, g3 = uint32_t(k) & 15u;
    S.tri[(k & ~15) | (g3 ^ g1 ^ tri_rot(g2))] =
        as_sel(stv16_compose(stv16_compose(S.delta[g1], S.delta[g2]), S.delta[g3]));
  }
  __syncthreads();
  const uint32_t n_warps = gridDim.x * WW;
  for (uint32_t p = blockIdx.x * WW + (t >> 5); p < P.n_pieces; p += n_warps) {
    const uint64_t c0 = uint64_t(p) * PIECE + uint64_t(lane) * CB;
    const uint32_t clen = chunk_len(c0, P.n);
    uint32_t w[16];
    load_chunk(P, c0, clen, w);
    Stv16 G = stv16_id();
    if (clen == CB) {  // back to front: bytes 61-63, 58-60, ..., 1-3, then byte 0
#pragma unroll
      for (int j = CB - 3; j >= 1; j -= 3)
        G = stv_step(G, at_byte(S.tri, S.ga[byte_of(w, j)] ^ S.gb[byte_of(w, j + 1)] ^
                                           S.gc[byte_of(w, j + 2)]));
      G = stv_step(G, at_byte(S.single, S.gc[byte_of(w, 0)]));
    } else {
      for (int j = int(clen) - 1; j >= 0; --j) G = stv_step(G, at_byte(S.single, S.gc[P.in[c0 + j]]));
    }
    Stv16 inc = G;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const Stv16 o = shfl_up16(inc, d);
      if (lane >= d) inc = stv16_compose(o, inc);
    }
    Stv16 ex = shfl_up16(inc, 1);
    if (lane == 0) ex = stv16_id();
    P.lane_pre[size_t(p) * 32 + lane] = stv16_pack(ex);
    if (lane == 31) P.piece_stv[p] = stv16_pack(inc);
  }
}

// ------------------------------------------------------------ pass 2
__global__ void __launch_bounds__(SCAN_T) tok_state_scan_kernel(const __grid_constant__ TokParams P) {
  __shared__ uint32_t tile_s;
  __shared__ Stv16 wv[SCAN_T / 32];
  __shared__ uint64_t pre_s[2];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) tile_s = atomicAdd(&P.tickets[0], 1u);
  __syncthreads();
  const uint32_t tile = tile_s;
  const uint64_t e0 = uint64_t(tile) * SCAN_TILE + uint64_t(t) * SCAN_E;
  uint64_t v[SCAN_E];
#pragma unroll
  for (int e = 0; e < SCAN_E; ++e) v[e] = e0 + e < P.n_pieces ? P.piece_stv[e0 + e] : 0ull;
  Stv16 acc = stv16_id();
#pragma unroll
  for (int e = 0; e < SCAN_E; ++e)
    if (e0 + e < P.n_pieces) acc = stv16_compose(acc, stv16_unpack(v[e]));
  Stv16 inc = acc;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Stv16 o = shfl_up16(inc, d);
    if (lane >= d) inc = stv16_compose(o, inc);
  }
  Stv16 lex = shfl_up16(inc, 1);
  if (lane == 0) lex = stv16_id();
  if (lane == 31) wv[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    constexpr int NWS = SCAN_T / 32;
    Stv16 wi = lane < NWS ? wv[lane] : stv16_id();
#pragma unroll
    for (int d = 1; d < NWS; d <<= 1) {
      const Stv16 o = shfl_up16(wi, d);
      if (lane >= d) wi = stv16_compose(o, wi);
    }
    Stv16 wex = shfl_up16(wi, 1);
    if (lane == 0) wex = stv16_id();
    Stv16 agg;
#pragma unroll
    for (int k = 0; k < 4; ++k) agg.w[k] = __shfl_sync(FULL, wi.w[k], NWS - 1);
    __syncwarp();
    if (lane < NWS) wv[lane] = wex;
    uint64_t a2[2], id2[2], ex2[2];
    stv16_to2(agg, a2);
    stv16_to2(stv16_id(), id2);
    lookback_vec<2>(P.flag_s, P.agg_s, P.inc_s, tile, a2, id2, id2, Stv16ComposeOp{},
                    LookbackCfg{P.st, P.spin_limit}, ex2);
    if (lane == 0) { pre_s[0] = ex2[0]; pre_s[1] = ex2[1]; }
  }
  __syncthreads();
  const uint64_t pre2[2] = {pre_s[0], pre_s[1]};
  uint32_t s = stv16_apply(stv16_from2(pre2), P.dfa.start_state);
  s = stv16_apply(wv[warp], s);
  s = stv16_apply(lex, s);
#pragma unroll
  for (int e = 0; e < SCAN_E; ++e) {
    if (e0 + e < P.n_pieces) {
      P.piece_state[e0 + e] = uint8_t(s);
      s = nib_apply(v[e], s);
    }
  }
}

// ------------------------------------------------------------ pass 3
// The count pass looks up two tables per byte, both replicated per lane:
// entry e is stored 32 times, lane l's copy at word e * 32 + l, so the 32
// lookups of a warp always fall in 32 different banks (one wavefront each,
// whatever the bytes and states).  Values are pre-shifted to be byte
// offsets: grp[b] = group * 2048, trans[g * 16 + s] = next * 128 | begin
// flag; the lane's copy adds lane * 4.  The state is carried as
// s * 128 | lane * 4.
constexpr int DT = 512;  // threads per block, count pass
constexpr int DW = DT / 32;
constexpr uint32_t R_NEXT = 0x780u, R_BEGIN_BIT = 11;

struct RepTables {
  uint32_t grp[256 * 32];
  uint32_t trans[256 * 32];
  uint8_t token_id[PP_MAX_STATES];
  uint8_t byte_token_id[256];
};

__device__ void build_rep_tables(const TokParams& P, RepTables& R) {
  const int t = threadIdx.x;
  for (int k = t; k < 256 * 32; k += blockDim.x) {
    const uint32_t e = uint32_t(k) >> 5;  // one entry per warp: uniform parameter reads
    R.grp[k] = (P.dfa.byte_to_group[e] & 0xFu) << 11;
    const uint32_t g = e >> 4, st = e & 0xFu;
    R.trans[k] = ((P.dfa.delta[g][st] & 0xFu) << 7) |
                 (P.dfa.tag[st][g] == PP_TAG_BEGIN ? 1u << R_BEGIN_BIT : 0u);
  }
  for (int k = t; k < 256; k += blockDim.x) R.byte_token_id[k] = P.dfa.byte_token_id[k];
  if (t < PP_MAX_STATES) R.token_id[t] = P.dfa.token_id[t];
}

__device__ __forceinline__ uint32_t lds_at(const uint32_t* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(base) + off);
}
// one DFA step on byte b; returns the begin flag
__device__ __forceinline__ uint32_t dfa_step(const RepTables& R, uint32_t b, uint32_t lane4,
                                             uint32_t& s) {
  const uint32_t v = lds_at(R.trans, lds_at(R.grp, (b << 7) | lane4) | s);
  s = (v & R_NEXT) | lane4;
  return (v >> R_BEGIN_BIT) & 1u;
}

// The DFA over the 32 bytes of half h of the chunk: returns the begin mask.
// With STATES, sn[4] gets the state before every byte as nibbles (byte j at
// bits 4(j & 7) of sn[j >> 3]).  PARTIAL: bytes at or past clen are skipped.
template <bool PARTIAL, bool STATES>
__device__ __forceinline__ uint32_t dfa_half(const RepTables& R, const uint32_t (&w)[16], int h,
                                             uint32_t clen, uint32_t lane4, uint32_t& s,
                                             uint32_t (&sn)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int jj = 32 * h + j;
    if (PARTIAL && uint32_t(jj) >= clen) break;
    if (STATES) sn[j >> 3] |= (s >> 7) << (4 * (j & 7));
    m |= dfa_step(R, byte_of(w, jj), lane4, s) << j;
  }
  return m;
}

// first transition into the invalid state in the chunk (slow path, only
// when the chunk starts valid and ends invalid; the invalid state absorbs)
__device__ uint32_t first_invalid(const TokParams& P, const RepTables& R, uint64_t c0,
                                  uint32_t clen, uint32_t lane4, uint32_t s) {
  const uint32_t inv = P.dfa.invalid_state;
  for (uint32_t j = 0; j < clen; ++j) {
    dfa_step(R, P.in[c0 + j], lane4, s);
    if ((s >> 7) == inv) return j;
  }
  return clen;
}

__global__ void __launch_bounds__(DT, 2) tok_count_kernel(const __grid_constant__ TokParams P) {
  extern __shared__ __align__(16) uint8_t dsm[];
  RepTables& R = *reinterpret_cast<RepTables*>(dsm);
  build_rep_tables(P, R);
  __syncthreads();
  const int t = threadIdx.x, lane = t & 31;
  const uint32_t lane4 = uint32_t(lane) * 4;
  const uint32_t inv = P.dfa.invalid_state;
  const uint32_t n_warps = gridDim.x * DW;
  for (uint32_t p = blockIdx.x * DW + (t >> 5); p < P.n_pieces; p += n_warps) {
    const uint64_t c0 = uint64_t(p) * PIECE + uint64_t(lane) * CB;
    const uint32_t clen = chunk_len(c0, P.n);
    const uint32_t s0 = nib_apply(P.lane_pre[size_t(p) * 32 + lane], P.piece_state[p]);
    uint32_t w[16];
    load_chunk(P, c0, clen, w);
    uint32_t s = (s0 << 7) | lane4, sn[4], m0, m1;
    if (clen == CB) {
      m0 = dfa_half<false, false>(R, w, 0, clen, lane4, s, sn);
      m1 = dfa_half<false, false>(R, w, 1, clen, lane4, s, sn);
    } else {
      m0 = dfa_half<true, false>(R, w, 0, clen, lane4, s, sn);
      m1 = dfa_half<true, false>(R, w, 1, clen, lane4, s, sn);
    }
    s >>= 7;
    if (c0 == 0 && clen > 0) m0 |= 1u;  // the first token starts at byte 0
    if (s == inv && s0 != inv)
      report(P.st, PP_ERR_INVALID_INPUT, c0 + first_invalid(P, R, c0, clen, lane4, (s0 << 7) | lane4),
             true);
    if (!P.carry_out && clen > 0 && c0 + clen == P.n && s != inv && !((P.dfa.accept_mask >> s) & 1u))
      report(P.st, PP_ERR_BAD_END_STATE, P.n, true);
    const uint32_t cnt = __popc(m0) + __popc(m1);
    const uint32_t last = m1 ? 64u - __clz(m1) : m0 ? 32u - __clz(m0) : 0u;
    P.lane_info[size_t(p) * 32 + lane] = s0 | (cnt << 4) | (last << 11);
    const uint32_t total = __reduce_add_sync(FULL, cnt);
    const uint32_t has = __ballot_sync(FULL, last != 0);
    const int ll = has ? 31 - __clz(has) : 0;
    const uint32_t l_last = __shfl_sync(FULL, last, ll);
    if (lane == 0) {
      P.piece_cnt[p] = total;
      P.piece_last[p] = has ? uint32_t(ll) * CB + l_last : 0u;
    }
  }
}

// ------------------------------------------------------------ pass 4
// (tokens, start + 1 of the last token start), combined earlier-then-later
struct CountOp {
  __device__ void operator()(const uint64_t (&a)[2], const uint64_t (&b)[2],
                             uint64_t (&o)[2]) const {
    o[0] = a[0] + b[0];
    o[1] = b[1] ? b[1] : a[1];
  }
};

__global__ void __launch_bounds__(SCAN_T) tok_count_scan_kernel(const __grid_constant__ TokParams P) {
  __shared__ uint32_t tile_s;
  __shared__ uint64_t wc[SCAN_T / 32], wl[SCAN_T / 32];
  __shared__ uint64_t pre_s[2];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) tile_s = atomicAdd(&P.tickets[1], 1u);
  __syncthreads();
  const uint32_t tile = tile_s;
  const uint64_t e0 = uint64_t(tile) * SCAN_TILE + uint64_t(t) * SCAN_E;
  uint32_t c[SCAN_E];
  uint64_t l[SCAN_E];
  uint64_t ac = 0, al = 0;
#pragma unroll
  for (int e = 0; e < SCAN_E; ++e) {
    const uint64_t idx = e0 + e;
    c[e] = 0;
    l[e] = 0;
    if (idx < P.n_pieces) {
      c[e] = P.piece_cnt[idx];
      const uint32_t r = P.piece_last[idx];
      l[e] = r ? idx * PIECE + r : 0ull;
    }
    ac += c[e];
    if (l[e]) al = l[e];
  }
  // warp and block scans
  uint64_t ic = ac, il = al;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t oc = __shfl_up_sync(FULL, ic, d), ol = __shfl_up_sync(FULL, il, d);
    if (lane >= d) { ic += oc; il = il ? il : ol; }
  }
  uint64_t xc = __shfl_up_sync(FULL, ic, 1), xl = __shfl_up_sync(FULL, il, 1);
  if (lane == 0) { xc = 0; xl = 0; }
  if (lane == 31) { wc[warp] = ic; wl[warp] = il; }
  __syncthreads();
  if (warp == 0) {
    constexpr int NWS = SCAN_T / 32;
    uint64_t vc = lane < NWS ? wc[lane] : 0ull, vl = lane < NWS ? wl[lane] : 0ull;
    uint64_t sc = vc, sl = vl;
#pragma unroll
    for (int d = 1; d < NWS; d <<= 1) {
      const uint64_t oc = __shfl_up_sync(FULL, sc, d), ol = __shfl_up_sync(FULL, sl, d);
      if (lane >= d) { sc += oc; sl = sl ? sl : ol; }
    }
    uint64_t ec = __shfl_up_sync(FULL, sc, 1), el = __shfl_up_sync(FULL, sl, 1);
    if (lane == 0) { ec = 0; el = 0; }
    const uint64_t a2[2] = {__shfl_sync(FULL, sc, NWS - 1), __shfl_sync(FULL, sl, NWS - 1)};
    __syncwarp();
    if (lane < NWS) { wc[lane] = ec; wl[lane] = el; }
    const uint64_t z[2] = {0ull, 0ull};
    uint64_t ex2[2];
    lookback_vec<2>(P.flag_c, P.agg_c, P.inc_c, tile, a2, z, z, CountOp{},
                    LookbackCfg{P.st, P.spin_limit}, ex2);
    if (lane == 0) { pre_s[0] = ex2[0]; pre_s[1] = ex2[1]; }
  }
  __syncthreads();
  uint64_t k = pre_s[0] + wc[warp] + xc;
  uint64_t pv = xl ? xl : wl[warp] ? wl[warp] : pre_s[1];
#pragma unroll
  for (int e = 0; e < SCAN_E; ++e) {
    const uint64_t idx = e0 + e;
    if (idx < P.n_pieces) {
      P.piece_k0[idx] = k;
      P.piece_prev[idx] = pv;
      k += c[e];
      if (l[e]) pv = l[e];
      if (idx + 1 == P.n_pieces) {
        P.st->n_tokens = k;
        if (P.carry_out) P.carry_out[0] = pv;
      }
    }
  }
}

// Partial mode: the DFA state before the last token start, re-run over the
// bytes of its chunk before it from the chunk's start state (one thread).
__global__ void tok_carry_kernel(const __grid_constant__ TokParams P) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const uint64_t ls1 = P.carry_out[0];
  if (ls1 == 0) { P.carry_out[1] = P.dfa.start_state; return; }
  const uint64_t ls = ls1 - 1, p = ls / PIECE;
  const uint32_t lane = uint32_t(ls % PIECE) / CB;
  uint32_t s = P.lane_info[size_t(p) * 32 + lane] & 0xFu;
  for (uint64_t j = p * PIECE + uint64_t(lane) * CB; j < ls; ++j)
    s = P.dfa.delta[P.dfa.byte_to_group[P.in[j]] & 0xFu][s] & 0xFu;
  P.carry_out[1] = s;
}

// ------------------------------------------------------------ pass 5 tables
// The DFA steps two bytes per lookup through composed pair transitions:
// pair[(g1 * 16 + g2) * 16 + s], addressed in bytes as g1 * 512 + g2 * 32 + 2s
// (the groups come from a byte table, so the 32 lanes' lookups of ASCII
// bytes fall in distinct banks),
// holds 2 x the state after both bytes (P2_NEXT2), the state between them
// (P2_MID), the token-begin flags of the two transitions (P2_BEGIN, first
// byte in the low bit) and their invalid flags (P2_INV).  The last chunk of
// the input steps one byte at a time through trans[g * 16 + s] = next state
// | T_BEGIN | T_INV.  An invalid flag marks a transition into the invalid
// state from another state.
constexpr uint32_t P2_NEXT2 = 0x1Eu, P2_MID = 0x1E0u, P2_BEGIN_SHIFT = 9, P2_INV = 0x1800u;
constexpr uint32_t T_BEGIN = 0x10u, T_INV = 0x20u;

struct DfaTables {
  uint8_t g8[256];      // group
  uint16_t pair[16 * 16 * 16];
  uint8_t grp16[256];   // group * 16
  uint8_t trans[256];
  uint8_t token_id[PP_MAX_STATES];
  uint8_t byte_token_id[256];
};

// one transition: next state | T_BEGIN | T_INV
__device__ __forceinline__ uint32_t trans_of(const TokParams& P, uint32_t g, uint32_t s) {
  const uint32_t nx = P.dfa.delta[g][s] & 0xFu;
  uint32_t e = nx;
  if (P.dfa.tag[s][g] == PP_TAG_BEGIN) e |= T_BEGIN;
  if (nx == P.dfa.invalid_state && s != P.dfa.invalid_state) e |= T_INV;
  return e;
}

__device__ void build_dfa_tables(const TokParams& P, DfaTables& S) {
  const int t = threadIdx.x;
  for (int k = t; k < 256; k += blockDim.x) {
    const uint32_t g = P.dfa.byte_to_group[k] & 0xFu;
    S.g8[k] = uint8_t(g);
    S.grp16[k] = uint8_t(g << 4);
    S.trans[k] = uint8_t(trans_of(P, uint32_t(k) >> 4, uint32_t(k) & 0xFu));
    S.byte_token_id[k] = P.dfa.byte_token_id[k];
  }
  for (int k = t; k < 16 * 16 * 16; k += blockDim.x) {
    const uint32_t g1 = uint32_t(k) >> 8, g2 = (uint32_t(k) >> 4) & 0xFu, s = uint32_t(k) & 0xFu;
    const uint32_t e1 = trans_of(P, g1, s), s1 = e1 & 0xFu;
    const uint32_t e2 = trans_of(P, g2, s1);
    S.pair[k] = uint16_t(((e2 & 0xFu) << 1) | (s1 << 5) |
                         ((e1 & T_BEGIN) ? 1u << P2_BEGIN_SHIFT : 0u) |
                         ((e2 & T_BEGIN) ? 2u << P2_BEGIN_SHIFT : 0u) |
                         (((e1 | e2) & T_INV) ? P2_INV : 0u));
  }
  if (t < PP_MAX_STATES) S.token_id[t] = P.dfa.token_id[t];
}

// One DFA over the 32 bytes of half h of a full chunk, two bytes a step:
// returns the begin mask; s2 is 2 x the state.  With STATES, sn[4] gets the
// state before every byte as nibbles (byte j at bits 4(j & 7) of sn[j >> 3]).
template <bool STATES>
__device__ __forceinline__ uint32_t dfa_pairs(const DfaTables& S, const uint32_t (&w)[16], int h,
                                              uint32_t& s2, uint32_t& any, uint32_t (&sn)[4]) {
  const uint8_t* tb = reinterpret_cast<const uint8_t*>(S.pair);
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int j = 32 * h + 2 * q;
    const uint32_t g1 = S.g8[byte_of(w, j)], g2 = S.g8[byte_of(w, j + 1)];
    const uint32_t v = *reinterpret_cast<const uint16_t*>(tb + ((g1 << 9) | (g2 << 5) | s2));
    if (STATES) sn[q >> 2] |= ((s2 | (v & P2_MID)) >> 1) << (8 * (q & 3));
    m |= ((v >> P2_BEGIN_SHIFT) & 3u) << (2 * q);
    any |= v;
    s2 = v & P2_NEXT2;
  }
  return m;
}

// The same one byte at a time for the last, partial chunk (bytes at or past
// clen leave the state and the mask alone); s is the state itself.
template <bool STATES>
__device__ __forceinline__ uint32_t dfa_bytes(const DfaTables& S, const uint32_t (&w)[16], int h,
                                              uint32_t clen, uint32_t& s, uint32_t& any,
                                              uint32_t (&sn)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int jj = 32 * h + j;
    if (uint32_t(jj) >= clen) break;
    if (STATES) sn[j >> 3] |= s << (4 * (j & 7));
    const uint32_t v = S.trans[S.grp16[byte_of(w, jj)] | s];
    m |= ((v >> 4) & 1u) << j;
    any |= v;
    s = v & 0xFu;
  }
  return m;
}

// ------------------------------------------------------------ pass 5
// A piece's token starts in order: offset in the piece and the state before
// the start (which gives the id of the token it closes).  Entry `total`
// holds the state after the last byte of the input, in the last piece.
struct EmitStage {
  uint16_t start[WW][CAPW];
  uint8_t state[WW][CAPW + 1];
};

__device__ __forceinline__ uint32_t nibble(const uint32_t (&sn)[4], uint32_t j) {
  const uint32_t x = j < 16 ? (j < 8 ? sn[0] : sn[1]) : (j < 24 ? sn[2] : sn[3]);
  return (x >> (4 * (j & 7))) & 0xFu;
}

// id of the token that starts at `start` and ends in state s_end
__device__ __forceinline__ uint32_t token_id(const TokParams& P, const DfaTables& S,
                                             uint32_t s_end, uint64_t start) {
  const uint32_t id = S.token_id[s_end];
  return id == 0xFEu ? S.byte_token_id[__ldg(P.in + start)] : id;
}

// One half of the chunk: run the DFA, return the begin mask and the states
// before every byte.
__device__ __forceinline__ uint32_t emit_half(const DfaTables& S, const uint32_t (&w)[16], int h,
                                              bool full, uint32_t clen, uint32_t& s,
                                              uint32_t (&sn)[4]) {
  uint32_t any = 0, m;
#pragma unroll
  for (int k = 0; k < 4; ++k) sn[k] = 0;
  if (full) {
    uint32_t s2 = 2 * s;
    m = dfa_pairs<true>(S, w, h, s2, any, sn);
    s = s2 >> 1;
  } else {
    m = dfa_bytes<true>(S, w, h, clen, s, any, sn);
  }
  return m;
}

__global__ void __launch_bounds__(WT, EMIT_BPS) tok_emit_kernel(const __grid_constant__ TokParams P) {
  __shared__ DfaTables S;
  __shared__ EmitStage E;
  build_dfa_tables(P, S);
  __syncthreads();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const bool sizing = P.cap == 0 && P.out_start == nullptr;
  const uint32_t n_warps = gridDim.x * WW;
  for (uint32_t p = blockIdx.x * WW + warp; p < P.n_pieces; p += n_warps) {
    const uint64_t pbase = uint64_t(p) * PIECE;
    const uint32_t off0 = uint32_t(lane) * CB;
    const uint64_t c0 = pbase + off0;
    const uint32_t clen = chunk_len(c0, P.n);
    const bool full = clen == CB;
    const bool owns_end = clen > 0 && c0 + clen == P.n;
    const uint32_t info = P.lane_info[size_t(p) * 32 + lane];
    const uint32_t cnt = (info >> 4) & 0x7Fu;
    const uint64_t k0 = P.piece_k0[p];
    uint32_t ib = cnt;  // the lane's first token, piece-local
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, ib, d);
      if (lane >= d) ib += o;
    }
    const uint32_t total = __shfl_sync(FULL, ib, 31);
    ib -= cnt;
    uint32_t w[16];
    load_chunk(P, c0, clen, w);
    uint32_t s = info & 0xFu;
    {  // the warp's next piece: towards L2 while this one is processed
      const uint64_t cn = c0 + uint64_t(n_warps) * PIECE;
      if (cn < P.n) asm volatile("prefetch.global.L2 [%0];" ::"l"(P.in + cn));
    }

    if (total <= CAPW) {
      // ---- stage the starts, then write all three arrays coalesced
      uint32_t i = ib;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sn[4];
        uint32_t m = emit_half(S, w, h, full, clen, s, sn);
        if (h == 0 && c0 == 0 && clen > 0) m |= 1u;  // the first token starts at byte 0
        while (m) {
          const uint32_t j = __ffs(m) - 1;
          m &= m - 1;
          E.start[warp][i] = uint16_t(off0 + 32 * h + j);
          E.state[warp][i] = uint8_t(nibble(sn, j));
          ++i;
        }
      }
      if (owns_end) E.state[warp][i] = uint8_t(s);
      __syncwarp();
      // starts of tokens k0 .. k0+total-1; lengths and ids of the tokens
      // they close, k0-1 .. k0+total-2, and of the last token in the last piece
      const uint64_t prev = P.piece_prev[p];  // start + 1 of the token open at the piece start
      const uint32_t nclose = total + (p + 1 == P.n_pieces && !P.carry_out ? 1u : 0u);
      if (k0 + nclose <= P.cap) {
        // every entry of the piece fits: piece offsets in 32 bits, the
        // previous start from the neighbouring lane
        const uint32_t n_rel = uint32_t(min(P.n - pbase, uint64_t(PIECE)));
        uint32_t carry = 0;  // the previous batch's last start (lane 31's), for lane 0
        for (uint32_t b = 0; b < nclose; b += 32) {
          const uint32_t q = b + uint32_t(lane);
          const uint32_t e = q < total ? uint32_t(E.start[warp][q]) : n_rel;
          uint32_t pe = __shfl_up_sync(FULL, e, 1);
          if (lane == 0) pe = carry;
          carry = __shfl_sync(FULL, e, 31);
          if (q < nclose) {
            if (q < total) P.out_start[k0 + q] = pbase + e;
            if (q > 0) {
              P.out_len[k0 + q - 1] = e - pe;
              P.out_id[k0 + q - 1] = uint8_t(token_id(P, S, E.state[warp][q], pbase + pe));
            } else if (k0 > 0) {  // the token open at the piece start
              const uint64_t beg = prev - 1;
              P.out_len[k0 - 1] = uint32_t(pbase + e - beg);
              P.out_id[k0 - 1] = uint8_t(token_id(P, S, E.state[warp][0], beg));
            }
          }
        }
      } else {
        for (uint32_t q = lane; q < nclose; q += 32) {
          const uint64_t k = k0 + q;
          const uint64_t end = q < total ? pbase + E.start[warp][q] : P.n;
          if (q < total) {
            if (k < P.cap) P.out_start[k] = end;
            else if (!sizing) report(P.st, PP_ERR_CAPACITY, 0, false);
          }
          if (k >= 1 && k - 1 < P.cap) {  // token k-1 exists (the first start closes none)
            const uint64_t beg = q > 0 ? pbase + E.start[warp][q - 1] : prev - 1;
            P.out_len[k - 1] = uint32_t(end - beg);
            P.out_id[k - 1] = uint8_t(token_id(P, S, E.state[warp][q], beg));
          }
        }
      }
      __syncwarp();
    } else {
      // ---- dense piece: every start writes its own triple entries
      const uint32_t last = (info >> 11) & 0x7Fu;
      uint64_t lp = last ? c0 + last : 0ull;  // positions grow with the lane: max = latest
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint64_t o = __shfl_up_sync(FULL, lp, d);
        if (lane >= d) lp = max(lp, o);
      }
      uint64_t prev = __shfl_up_sync(FULL, lp, 1);  // start + 1 of the open token
      if (lane == 0) prev = 0;
      if (prev == 0) prev = P.piece_prev[p];
      uint64_t k = k0 + ib;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sn[4];
        uint32_t m = emit_half(S, w, h, full, clen, s, sn);
        if (h == 0 && c0 == 0 && clen > 0) m |= 1u;
        while (m) {
          const uint32_t j = __ffs(m) - 1;
          m &= m - 1;
          const uint64_t pos = c0 + 32 * h + j;
          if (prev && k - 1 < P.cap) {
            P.out_id[k - 1] = uint8_t(token_id(P, S, nibble(sn, j), prev - 1));
            P.out_len[k - 1] = uint32_t(pos - (prev - 1));
          }
          if (k < P.cap) P.out_start[k] = pos;
          else if (!sizing) report(P.st, PP_ERR_CAPACITY, 0, false);
          ++k;
          prev = pos + 1;
        }
      }
      if (!P.carry_out && owns_end && prev && k - 1 < P.cap) {  // close the last token
        P.out_id[k - 1] = uint8_t(token_id(P, S, s, prev - 1));
        P.out_len[k - 1] = uint32_t(P.n - (prev - 1));
      }
    }
  }
}

__global__ void tok_init_kernel(uint4* zero, size_t n16, pp_status* st) {
  const size_t i0 = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < n16; i += size_t(gridDim.x) * blockDim.x) zero[i] = make_uint4(0, 0, 0, 0);
  if (i0 == 0) {
    st->error = 0;
    st->reserved = 0;
    st->first_error_offset = ~0ull;
    st->n_records = 0;
    st->n_tokens = 0;
    for (int c = 0; c < PP_MAX_COLS; ++c) st->chars_len[c] = 0;
    st->n_dropped = 0;
  }
}

// ------------------------------------------------------------ host
size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
uint32_t pieces_of(uint64_t n) { return uint32_t((n + PIECE - 1) / PIECE); }
uint32_t scan_tiles_of(uint32_t pieces) { return (pieces + SCAN_TILE - 1) / SCAN_TILE; }

// [tickets 16][flag_s 4T][flag_c 4T] is zeroed by tok_init_kernel
size_t zeroed_bytes(uint32_t tiles) { return (16 + size_t(tiles) * 8 + 15) & ~size_t(15); }

struct Layout {
  size_t agg_s, inc_s, agg_c, inc_c, lane_pre, piece_stv, piece_state, lane_info, piece_cnt,
      piece_last, piece_k0, piece_prev, total;
};
Layout layout_of(uint64_t n) {
  const uint32_t P = pieces_of(n), T = scan_tiles_of(P);
  Layout L;
  size_t o = al256(zeroed_bytes(T));
  L.agg_s = o; o += al256(size_t(T) * 16);
  L.inc_s = o; o += al256(size_t(T) * 16);
  L.agg_c = o; o += al256(size_t(T) * 16);
  L.inc_c = o; o += al256(size_t(T) * 16);
  L.lane_pre = o; o += al256(size_t(P) * 32 * 8);
  L.piece_stv = o; o += al256(size_t(P) * 8);
  L.piece_state = o; o += al256(size_t(P));
  L.lane_info = o; o += al256(size_t(P) * 32 * 4);
  L.piece_cnt = o; o += al256(size_t(P) * 4);
  L.piece_last = o; o += al256(size_t(P) * 4);
  L.piece_k0 = o; o += al256(size_t(P) * 8);
  L.piece_prev = o; o += al256(size_t(P) * 8);
  L.total = o;
  return L;
}

}  // namespace

namespace ppi {

extern uint32_t g_spin_limit;

size_t tokenize_scratch_bytes(uint64_t n) { return layout_of(n).total; }

cudaError_t launch_tokenize(const uint8_t* in, uint64_t n, const GenericDfa& dfa,
                            uint8_t* out_id, uint64_t* out_start, uint32_t* out_len,
                            uint64_t cap, pp_status* st, void* scratch, size_t,
                            cudaStream_t stream, unsigned long long* carry_out) {
  TokParams P{};
  P.in = in;
  P.n = n;
  P.n_pieces = pieces_of(n);
  P.spin_limit = g_spin_limit;
  P.aligned = (reinterpret_cast<uintptr_t>(in) & 15) == 0;
  P.dfa = dfa;
  P.out_id = out_id;
  P.out_start = out_start;
  P.out_len = out_len;
  P.cap = cap;
  P.st = st;
  P.carry_out = carry_out;
  const uint32_t T = scan_tiles_of(P.n_pieces);
  const Layout L = layout_of(n);
  uint8_t* b = static_cast<uint8_t*>(scratch);
  P.tickets = reinterpret_cast<uint32_t*>(b);
  P.flag_s = reinterpret_cast<uint32_t*>(b + 16);
  P.flag_c = reinterpret_cast<uint32_t*>(b + 16 + size_t(T) * 4);
  P.agg_s = reinterpret_cast<uint64_t*>(b + L.agg_s);
  P.inc_s = reinterpret_cast<uint64_t*>(b + L.inc_s);
  P.agg_c = reinterpret_cast<uint64_t*>(b + L.agg_c);
  P.inc_c = reinterpret_cast<uint64_t*>(b + L.inc_c);
  P.lane_pre = reinterpret_cast<uint64_t*>(b + L.lane_pre);
  P.piece_stv = reinterpret_cast<uint64_t*>(b + L.piece_stv);
  P.piece_state = b + L.piece_state;
  P.lane_info = reinterpret_cast<uint32_t*>(b + L.lane_info);
  P.piece_cnt = reinterpret_cast<uint32_t*>(b + L.piece_cnt);
  P.piece_last = reinterpret_cast<uint32_t*>(b + L.piece_last);
  P.piece_k0 = reinterpret_cast<uint64_t*>(b + L.piece_k0);
  P.piece_prev = reinterpret_cast<uint64_t*>(b + L.piece_prev);

  const bool timed = stage_begin();
  if (timed) stage_mark(0, stream);
  const size_t n16 = zeroed_bytes(T) / 16;
  tok_init_kernel<<<int(std::min<size_t>((n16 + 255) / 256 + 1, 1024)), 256, 0, stream>>>(
      reinterpret_cast<uint4*>(b), n16, st);
  cudaError_t e = cudaGetLastError();
  if (timed) stage_mark(1, stream);
  if (e != cudaSuccess || P.n_pieces == 0) return e;
  int n_sm = 0, dev = 0;
  if ((e = sm_count(&n_sm)) != cudaSuccess) return e;
  if ((e = current_device(&dev)) != cudaSuccess) return e;
  static DeviceOnce attrs;
  e = attrs.run(dev, [](int) {
    return cudaFuncSetAttribute(tok_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(sizeof(RepTables)));
  });
  if (e != cudaSuccess) return e;
  const uint32_t bgrid = std::min<uint32_t>((P.n_pieces + WW - 1) / WW, uint32_t(n_sm) * 4);
  const uint32_t egrid = std::min<uint32_t>((P.n_pieces + WW - 1) / WW, uint32_t(n_sm) * EMIT_BPS);
  const uint32_t dgrid = std::min<uint32_t>((P.n_pieces + DW - 1) / DW, uint32_t(n_sm) * 2);
  tok_stv_kernel<<<bgrid, WT, 0, stream>>>(P);
  if (timed) stage_mark(2, stream);
  tok_state_scan_kernel<<<T, SCAN_T, 0, stream>>>(P);
  if (timed) stage_mark(3, stream);
  tok_count_kernel<<<dgrid, DT, sizeof(RepTables), stream>>>(P);
  if (timed) stage_mark(4, stream);
  tok_count_scan_kernel<<<T, SCAN_T, 0, stream>>>(P);
  if (carry_out) tok_carry_kernel<<<1, 32, 0, stream>>>(P);
  if (timed) stage_mark(5, stream);
  const bool sizing = cap == 0 && out_start == nullptr;
  if (!sizing) tok_emit_kernel<<<egrid, WT, 0, stream>>>(P);
  if (timed) stage_mark(6, stream);
  return cudaGetLastError();
}

}  // namespace ppi
