// State-transition vectors of a DFA with up to 16 states (ParPaRaw
// Section 3.1, Figure 2): lane s holds the state reached from start state s.
//
// In registers a vector is 16 byte lanes in four words (Stv16); stored, it
// is 16 nibbles in one uint64.  Lane values are below 16, so bit 7 of every
// byte is clear, which the byte permutes below rely on.
#pragma once
#include <cstdint>

#include "pp_device.cuh"

namespace ppd {

struct Stv16 { uint32_t w[4]; };

__device__ __forceinline__ Stv16 stv16_id() {
  return {{0x03020100u, 0x07060504u, 0x0B0A0908u, 0x0F0E0D0Cu}};
}

// Byte permute (PTX prmt, default mode).  Selector nibble k picks byte
// (nibble & 7) of {b, a} for output byte k; when the nibble's bit 3 is set
// the output byte is instead that byte's sign bit replicated, so 0x00 for
// any byte below 0x80.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four lanes of G picked by the selector nibbles (each 0..15): lanes 0-7
// come from the low pool, where nibbles >= 8 give 0, and lanes 8-15 from
// the high pool with the selector's bit 3 flipped.
__device__ __forceinline__ uint32_t stv16_gather(const Stv16& g, uint32_t sel, uint32_t sel_x) {
  return prmt(g.w[0], g.w[1], sel) | prmt(g.w[2], g.w[3], sel_x);
}

// (a o b)[i] = b[a[i]]: a is the earlier vector.
__device__ __forceinline__ Stv16 stv16_compose(const Stv16& a, const Stv16& b) {
  Stv16 r;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t v = a.w[k];
    const uint32_t sel = prmt(v | (v >> 4), 0u, 0x0020u);  // nibble j = a[4k + j]
    r.w[k] = stv16_gather(b, sel, sel ^ 0x8888u);
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

// 16 byte lanes <-> 16 nibbles (lane s at bits 4s..4s+3)
__device__ __forceinline__ uint64_t stv16_pack(const Stv16& g) {
  uint32_t x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = g.w[k] | (g.w[k] >> 4);  // bytes 0 and 2 hold lane pairs
  const uint32_t lo = prmt(x[0], x[1], 0x6420u), hi = prmt(x[2], x[3], 0x6420u);
  return uint64_t(lo) | (uint64_t(hi) << 32);
}
__device__ __forceinline__ Stv16 stv16_unpack(uint64_t v) {
  Stv16 g;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t x = uint32_t(v >> (32 * h));
    const uint32_t ev = x & 0x0F0F0F0Fu, od = (x >> 4) & 0x0F0F0F0Fu;
    g.w[2 * h] = prmt(ev, od, 0x5140u);
    g.w[2 * h + 1] = prmt(ev, od, 0x7362u);
  }
  return g;
}
__device__ __forceinline__ uint32_t nib_apply(uint64_t v, uint32_t s) {
  return uint32_t(v >> (4 * s)) & 0xFu;
}

// Composition on the two-word form used by the look-back (lanes 0-7 in
// word 0, 8-15 in word 1, bytes as in Stv16).
struct Stv16ComposeOp {
  __device__ void operator()(const uint64_t (&a)[2], const uint64_t (&b)[2],
                             uint64_t (&o)[2]) const {
    const Stv16 A = {{uint32_t(a[0]), uint32_t(a[0] >> 32), uint32_t(a[1]), uint32_t(a[1] >> 32)}};
    const Stv16 B = {{uint32_t(b[0]), uint32_t(b[0] >> 32), uint32_t(b[1]), uint32_t(b[1] >> 32)}};
    const Stv16 R = stv16_compose(A, B);
    o[0] = uint64_t(R.w[0]) | (uint64_t(R.w[1]) << 32);
    o[1] = uint64_t(R.w[2]) | (uint64_t(R.w[3]) << 32);
  }
};
__device__ __forceinline__ void stv16_to2(const Stv16& g, uint64_t (&o)[2]) {
  o[0] = uint64_t(g.w[0]) | (uint64_t(g.w[1]) << 32);
  o[1] = uint64_t(g.w[2]) | (uint64_t(g.w[3]) << 32);
}
__device__ __forceinline__ Stv16 stv16_from2(const uint64_t (&a)[2]) {
  return {{uint32_t(a[0]), uint32_t(a[0] >> 32), uint32_t(a[1]), uint32_t(a[1] >> 32)}};
}

}  // namespace ppd
