// General-DFA kernel (|S| <= 16) on sm_103a: pp_tags, the per-byte state
// and tag of any DFA (a test hook for the scan machinery; pp_tokenize has
// its own passes).
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
#include <cstdint>
#include <cuda_runtime.h>
#include <algorithm>

#include "pp.h"
#include "pp_device.cuh"
#include "pp_internal.h"
#include "pp_stv16.cuh"

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
struct SharedG {
  uint32_t tile;
  uint32_t pad;
  uint64_t pre[2];
  Stv16 warp_stv[NW];
  GroupOps ops[PP_MAX_GROUPS];
  uint8_t grp[256];
  uint8_t delta[PP_MAX_GROUPS * PP_MAX_STATES];  // [group][state]
  uint8_t tag[PP_MAX_STATES * PP_MAX_GROUPS];    // [state][group]
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
  pp_status* st;
  uint32_t* tile_counter;
  uint32_t* lb1_flag;
  uint64_t* lb1_agg;
  uint64_t* lb1_inc;
};

__device__ void setup_tables(const GParams& P, SharedG& S) {
  const int t = threadIdx.x;
  for (int k = t; k < 256; k += NT) {
    S.grp[k] = P.dfa.byte_to_group[k];
  }
  for (int k = t; k < PP_MAX_GROUPS * PP_MAX_STATES; k += NT) {
    S.delta[k] = (&P.dfa.delta[0][0])[k];
    S.tag[k] = (&P.dfa.tag[0][0])[k];
  }
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
    lookback_vec<2>(P.lb1_flag, P.lb1_agg, P.lb1_inc, tile, a2, i2, i2, Stv16ComposeOp{}, cfg, ex);
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
    st->n_dropped = 0;
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

// [counter 16][lb1_flag 4n] zeroed, then lb1_agg/inc (16n each)
size_t zero_bytes(uint32_t n) { return (16 + size_t(n) * 4 + 15) & ~size_t(15); }

void carve(void* base, uint32_t n, GParams& P) {
  uint8_t* p = static_cast<uint8_t*>(base);
  P.tile_counter = reinterpret_cast<uint32_t*>(p);
  P.lb1_flag = reinterpret_cast<uint32_t*>(p + 16);
  p += align256(zero_bytes(n));
  P.lb1_agg = reinterpret_cast<uint64_t*>(p); p += align256(size_t(n) * 16);
  P.lb1_inc = reinterpret_cast<uint64_t*>(p);
}

uint32_t n_tiles_of(uint64_t n) { return uint32_t((n + TILE - 1) / TILE); }

cudaError_t run(void (*kern)(GParams), size_t dyn_smem, const GParams& P, void* scratch,
                cudaStream_t stream) {
  const size_t n16 = zero_bytes(P.n_tiles) / 16;
  generic_init_kernel<<<int(std::min<size_t>((n16 + 255) / 256 + 1, 1024)), 256, 0, stream>>>(
      static_cast<uint4*>(scratch), n16, P.st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || P.n_tiles == 0) return e;
  int n_sm = 0;
  if ((e = ppi::sm_count(&n_sm)) != cudaSuccess) return e;
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
  return align256(zero_bytes(nt)) + 2 * align256(size_t(nt) * 16);
}

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

cudaError_t launch_count_byte(const uint8_t* in, uint64_t n, uint8_t value, uint64_t* d_count,
                              cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(d_count, 0, sizeof(uint64_t), stream);
  if (e != cudaSuccess || n == 0) return e;
  int n_sm = 0;
  if ((e = ppi::sm_count(&n_sm)) != cudaSuccess) return e;
  const uint64_t want = (n / 16 + 255) / 256;
  const int blocks = int(std::min<uint64_t>(want ? want : 1, uint64_t(n_sm) * 8));
  count_byte_kernel<<<blocks, 256, 0, stream>>>(in, n, value, d_count);
  return cudaGetLastError();
}

}  // namespace ppi
