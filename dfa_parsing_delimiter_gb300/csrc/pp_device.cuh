// Device-side building blocks shared by the libpp kernels (sm_103a).
//
//  * memory-order primitives for the cross-block scan (release/acquire at
//    GPU scope, L2-only payload loads),
//  * a warp-cooperative, single-pass decoupled look-back over an arbitrary
//    associative operation, with a bounded wait (the cross-block exclusive
//    scan of ParPaRaw Sections 3.1/3.2: "an exclusive scan using the
//    composite operation" and the scans of record counts / column offsets),
//  * helpers for 4-lane state-transition vectors held as bytes in one
//    32-bit register (ParPaRaw Section 3.1, Figure 2).
#pragma once
#include <cstdint>
#include "pp.h"

namespace ppd {

constexpr unsigned FULL = 0xFFFFFFFFu;

// ------------------------------------------------------------- memory order
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// status updates (device-side error reporting, never a trap)
__device__ __forceinline__ void report(pp_status* st, int bit, uint64_t off, bool with_off) {
  atomicOr(&st->error, bit);
  if (with_off) atomicMin(reinterpret_cast<unsigned long long*>(&st->first_error_offset),
                          static_cast<unsigned long long>(off));
}

// --------------------------------------------------------------- STV, 4 lanes
// A state-transition vector over states 0..3 lives in one register, entry i
// in byte i.  State 4 (if the DFA has it) is an absorbing invalid state; it
// is not stored: the second PRMT source supplies it (0x04 in every byte).
constexpr uint32_t STV_ID = 0x03020100u;
constexpr uint32_t STV_INV_POOL = 0x04040404u;

// bytes v0..v3 (each <= 4) -> PRMT selector nibbles v0 | v1<<4 | v2<<8 | v3<<12
__device__ __forceinline__ uint32_t stv_as_selector(uint32_t a) {
  uint32_t x = a | (a >> 4);
  return __byte_perm(x, 0, 0x0020);
}
// composite: (a o b)[i] = b[a[i]]  (a = earlier chunk, b = later chunk)
__device__ __forceinline__ uint32_t stv_compose(uint32_t a, uint32_t b) {
  return __byte_perm(b, STV_INV_POOL, stv_as_selector(a));
}
// v[s] (s <= 4; s == 4 stays 4)
__device__ __forceinline__ uint32_t stv_apply(uint32_t v, uint32_t s) {
  return s >= 4 ? 4u : (v >> (8 * s)) & 0xFFu;
}

// ------------------------------------------------------------ look-back
// Tile-state flags.
constexpr uint32_t LB_NONE = 0, LB_AGG = 1, LB_INC = 2;

struct LookbackCfg {
  pp_status* st;
  uint32_t spin_limit;  // polls before giving up with PP_ERR_LOOKBACK_TIMEOUT
};

// The window is usable once every lane up to (and including) the nearest
// predecessor that published an inclusive prefix has published something;
// lanes further back are not needed.
__device__ __forceinline__ bool lb_ready(uint32_t f) {
  const uint32_t inc = __ballot_sync(FULL, f == LB_INC);
  const uint32_t none = __ballot_sync(FULL, f == LB_NONE);
  const uint32_t below = inc ? ((inc & (0u - inc)) - 1u) : FULL;
  return (none & below) == 0;
}

// Bounded poll: returns false when the limit is exhausted.
__device__ __forceinline__ bool lb_backoff(uint32_t& spins, uint32_t limit) {
  if (++spins > limit) return false;
  __nanosleep(spins < 64 ? 32 : 256);
  return true;
}

// Single-word look-back for 32-bit values packed with the flag into a u64:
// bits 62..63 = flag, bits 0..31 = value.  Executed by one full warp.
// Returns the exclusive prefix of `tile`, combining with op(earlier, later).
template <class Op>
__device__ uint32_t lookback_word(unsigned long long* words, uint32_t tile, uint32_t agg,
                                  uint32_t seed, uint32_t identity, Op op,
                                  const LookbackCfg& cfg) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
    if (lane == 0) st_relaxed64(&words[0], (uint64_t(LB_INC) << 62) | op(seed, agg));
    return seed;
  }
  if (lane == 0) st_relaxed64(&words[tile], (uint64_t(LB_AGG) << 62) | agg);
  uint32_t acc = identity;
  int64_t base = int64_t(tile) - 1;
  uint32_t spins = 0;
  bool timed_out = false;
  for (;;) {
    const int64_t idx = base - lane;
    uint64_t w;
    for (;;) {
      w = idx >= 0 ? ld_relaxed64(&words[idx]) : ((uint64_t(LB_INC) << 62) | seed);
      if (lb_ready(uint32_t(w >> 62))) break;
      if (!lb_backoff(spins, cfg.spin_limit)) {
        timed_out = true;
        if ((w >> 62) == LB_NONE) w = (uint64_t(LB_INC) << 62) | identity;
        break;
      }
    }
    const uint32_t f = uint32_t(w >> 62);
    const uint32_t v = uint32_t(w);
    const uint32_t pmask = __ballot_sync(FULL, f == LB_INC);
    const int stop = pmask ? __ffs(pmask) - 1 : 31;
    uint32_t r = lane <= stop ? v : identity;
    // lane L combines with lane L+d, which holds an EARLIER tile
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint32_t o = __shfl_down_sync(FULL, r, d);
      if (lane + d < 32) r = op(o, r);
    }
    r = __shfl_sync(FULL, r, 0);
    acc = op(r, acc);
    if (pmask) break;
    base -= 32;
  }
  if (timed_out && lane == 0) report(cfg.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
  if (lane == 0) st_relaxed64(&words[tile], (uint64_t(LB_INC) << 62) | op(acc, agg));
  return acc;
}

// Multi-word look-back: per tile a flag word plus two payload slots (the
// tile's own aggregate and its inclusive prefix), each K x uint64.  The
// payload is written with L2-only stores before a release store of the
// flag; readers acquire the flag, then read the payload from L2.
//
// lb_publish_vec posts the tile's aggregate (tile 0: its inclusive prefix)
// and returns at once; lb_resolve_vec later walks back over predecessors
// and posts the inclusive prefix.  Splitting the two lets a block do other
// work while its predecessors finish.  Both are executed by one full warp;
// `agg`, `seed`, `identity` and the result are K words replicated in every
// lane.
template <int K, class Op>
__device__ __forceinline__ void lb_publish_vec(uint32_t* flags, uint64_t* agg_arr,
                                               uint64_t* inc_arr, uint32_t tile,
                                               const uint64_t (&agg)[K],
                                               const uint64_t (&seed)[K], Op op) {
  if ((threadIdx.x & 31) != 0) return;
  uint64_t v[K];
  op(seed, agg, v);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    uint64_t* dst = (tile == 0 ? inc_arr : agg_arr) + size_t(tile) * K + k;
    __stcg(reinterpret_cast<unsigned long long*>(dst), tile == 0 ? v[k] : agg[k]);
  }
  st_release(&flags[tile], tile == 0 ? LB_INC : LB_AGG);
}

template <int K, class Op>
__device__ void lb_resolve_vec(uint32_t* flags, uint64_t* agg_arr, uint64_t* inc_arr,
                               uint32_t tile, const uint64_t (&agg)[K],
                               const uint64_t (&seed)[K], const uint64_t (&identity)[K], Op op,
                               const LookbackCfg& cfg, uint64_t (&out_excl)[K]) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) out_excl[k] = seed[k];
    return;
  }
  uint64_t acc[K];
#pragma unroll
  for (int k = 0; k < K; ++k) acc[k] = identity[k];
  int64_t base = int64_t(tile) - 1;
  uint32_t spins = 0;
  bool timed_out = false;
  for (;;) {
    const int64_t idx = base - lane;
    uint32_t f;
    for (;;) {
      f = idx >= 0 ? ld_acquire(&flags[idx]) : LB_INC;
      if (lb_ready(f)) break;
      if (!lb_backoff(spins, cfg.spin_limit)) { timed_out = true; break; }
    }
    uint64_t v[K];
    if (idx < 0) {
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] = seed[k];
    } else if (f == LB_NONE) {  // only after a timeout
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] = identity[k];
      f = LB_INC;
    } else {
      const uint64_t* src = (f == LB_INC ? inc_arr : agg_arr) + size_t(idx) * K;
#pragma unroll
      for (int k = 0; k < K; ++k)
        v[k] = __ldcg(reinterpret_cast<const unsigned long long*>(src + k));
    }
    const uint32_t pmask = __ballot_sync(FULL, f == LB_INC);
    const int stop = pmask ? __ffs(pmask) - 1 : 31;
    if (lane > stop) {
#pragma unroll
      for (int k = 0; k < K; ++k) v[k] = identity[k];
    }
    // lane L combines with lane L+d, which holds an EARLIER tile
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint64_t o[K], t[K];
#pragma unroll
      for (int k = 0; k < K; ++k) o[k] = __shfl_down_sync(FULL, v[k], d);
      if (lane + d < 32) {
        op(o, v, t);
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] = t[k];
      }
    }
    uint64_t r[K], t[K];
#pragma unroll
    for (int k = 0; k < K; ++k) r[k] = __shfl_sync(FULL, v[k], 0);
    op(r, acc, t);
#pragma unroll
    for (int k = 0; k < K; ++k) acc[k] = t[k];
    if (pmask) break;
    base -= 32;
  }
  if (timed_out && lane == 0) report(cfg.st, PP_ERR_LOOKBACK_TIMEOUT, 0, false);
  uint64_t inc[K];
  op(acc, agg, inc);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k)
      __stcg(reinterpret_cast<unsigned long long*>(&inc_arr[size_t(tile) * K + k]), inc[k]);
    st_release(&flags[tile], LB_INC);
  }
#pragma unroll
  for (int k = 0; k < K; ++k) out_excl[k] = acc[k];
}

// Publish and resolve in one go.
template <int K, class Op>
__device__ void lookback_vec(uint32_t* flags, uint64_t* agg_arr, uint64_t* inc_arr,
                             uint32_t tile, const uint64_t (&agg)[K], const uint64_t (&seed)[K],
                             const uint64_t (&identity)[K], Op op, const LookbackCfg& cfg,
                             uint64_t (&out_excl)[K]) {
  lb_publish_vec<K>(flags, agg_arr, inc_arr, tile, agg, seed, op);
  __syncwarp();
  lb_resolve_vec<K>(flags, agg_arr, inc_arr, tile, agg, seed, identity, op, cfg, out_excl);
}

// ------------------------------------------------ 1-D bulk copy (TMA engine)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// one arrival that also announces `bytes` of asynchronous transfer
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(64);
  }
  return mbar_try_wait(bar, parity);
}
// Start moving the 128-byte line at p towards L2 (a hint; no result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Global -> shared bulk copy completed on `bar` (dst, src 16-byte aligned,
// bytes a multiple of 16).  Orders the CTA's earlier generic-proxy accesses
// of dst before the asynchronous write.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// x << n for 0 <= n <= 32 (PTX clamps shift amounts to the register width,
// so n == 32 gives 0)
__device__ __forceinline__ uint32_t shl32(uint32_t x, uint32_t n) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(n));
  return r;
}
// bits [a, b) of a 32-bit mask, 0 <= a <= b <= 32
__device__ __forceinline__ uint32_t range_mask(uint32_t a, uint32_t b) {
  return shl32(0xFFFFFFFFu, a) & ~shl32(0xFFFFFFFFu, b);
}

}  // namespace ppd
