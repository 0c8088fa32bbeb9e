// pp_parse_noalloc: pp_parse with its cross-tile scratch in a fixed
// buffer compiled into the library, so a call allocates no device memory.
//
// Who needs it: pp_parse takes its scratch from the stream-ordered
// allocator (cudaMallocAsync on the caller's stream).  Some callers cannot
// allocate there: processes on a device or driver set-up without
// stream-ordered memory pools (cudaDevAttrMemoryPoolsSupported is 0, e.g.
// some virtualised or shared-GPU set-ups), where cudaMallocAsync fails;
// and services that fix their device memory at start-up (a hard memory
// budget, or a pool sized once and never grown), where an allocation in the
// request path can fail under memory pressure or has to be accounted for.
// Such callers use this entry point with inputs up to the buffer's limit.
//
// The buffer is a file-scope __device__ array, which exists once in every
// device context that loads this library's device code.  Its address is
// looked up once per device (cudaGetSymbolAddress) on the first call made
// on that device; later calls reuse it.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_internal.h"

static __device__ __align__(256) uint8_t pp_noalloc_scratch[PP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::atomic<void*> g_scratch_addr[MAX_DEVICES];

// Address of the buffer in the current device's context (set-up on first use).
pp_rc scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return PP_ECUDA;
  if (dev < 0 || dev >= MAX_DEVICES) return PP_EINVAL;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, pp_noalloc_scratch);
    if (e != cudaSuccess || !p) return PP_ECUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PP_OK;
}

}  // namespace

extern "C" {

pp_rc pp_parse_noalloc(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                       const pp_coltype* col_types, int32_t* const out_offsets[],
                       uint8_t* const out_chars[], void* const out_typed[],
                       size_t records_capacity, const size_t chars_capacity[],
                       pp_status* d_status, cudaStream_t stream) {
  ppi::ParseParams p;
  pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, n_cols, col_types, out_offsets, out_chars,
                                out_typed, records_capacity, chars_capacity, d_status, &p);
  if (rc != PP_OK) return rc;
  const int ns = ppi::parse_ns_width(p.n_str);
  const size_t sb = ppi::parse_scratch_bytes(p.n_tiles, ns, p.enc != 0);
  if (sb > PP_NOALLOC_SCRATCH_BYTES) return PP_ETOOLARGE;  // before any CUDA call
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != PP_OK) return rc;
  // The tile counters and look-back flags, the only parts of the buffer
  // that must start at zero, are zeroed by the first kernel launch_parse
  // enqueues; every other byte is written before it is read.
  ppi::parse_scratch_carve(scratch, p.n_tiles, ns, &p.s, p.enc != 0);
  const cudaError_t e = ppi::launch_parse(p, stream);
  if (e == cudaSuccess) return PP_OK;
  return e == cudaErrorMemoryAllocation ? PP_ENOMEM : PP_ECUDA;
}

}  // extern "C"
