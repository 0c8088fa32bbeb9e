// pp_parse_host: pp_parse of an input in host memory into outputs in host
// memory, streamed through the device in chunks so that the copies in both
// directions overlap the parse (ParPaRaw Section 4, the streaming set-up:
// the input moves to the device in partitions while earlier partitions are
// parsed and their results move back).
//
// Per chunk i, on the caller's stream (cs) unless noted:
//   h2d stream:   new bytes of chunk i+1, host -> device staging buffer
//   cs:           input i = bytes carried over from chunk i-1 ++ staged bytes;
//                 pp_parse in partial mode (all but the last chunk): the
//                 unfinished record at the chunk end is not closed, and the
//                 end of the last complete record is reported;
//                 offsets rebased by the chars already emitted;
//                 chunk summary (status, record end, chars) -> host
//   host:         waits for the summary, merges the status, and carries the
//                 unfinished record (bytes after the last record delimiter)
//                 to the front of chunk i+1's input
//   d2h stream:   chunk i's complete records, device -> host outputs
// Two sets of device buffers alternate between chunks; the two copy
// directions run on their own streams, so both copy engines work at once.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_internal.h"

namespace {

using ppi::MAX_STR_COLS;

// Device summary of one chunk, copied to the host after its parse.
struct ChunkInfo {
  pp_status st;
  unsigned long long record_end;   // 1 + the chunk's last record delimiter (0: none)
  uint64_t chars[MAX_STR_COLS];    // chars of the chunk's complete records per string column
};

struct RebaseArgs {
  int32_t* off[MAX_STR_COLS];
  int64_t base[MAX_STR_COLS];
  int n_str;
  ChunkInfo* ci;
};

// Records the chars of the chunk's complete records (offsets[n_records])
// and adds the chars emitted by earlier chunks to offsets[1..n_records].
// The host has checked that the sums fit in int32.
__global__ void rebase_kernel(RebaseArgs a) {
  const uint64_t n = a.ci->st.n_records;
  const uint64_t i0 = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (int si = 0; si < a.n_str; ++si) {
    int32_t* o = a.off[si];
    if (n == 0) {
      if (i0 == 0) a.ci->chars[si] = 0;
      continue;
    }
    for (uint64_t i = 1 + i0; i <= n; i += stride) {  // entry n is read and rebased by one thread
      const int32_t v = o[i];
      if (i == n) a.ci->chars[si] = uint64_t(uint32_t(v));
      o[i] = int32_t(int64_t(v) + a.base[si]);
    }
  }
}

size_t width_of(int ty) {
  switch (ty) {
    case PP_COL_INT8: return 1;
    case PP_COL_INT32: return 4;
    case PP_COL_INT64: case PP_COL_FLOAT64: return 8;
    default: return 0;
  }
}

pp_rc rc_of(cudaError_t e) {
  if (e == cudaSuccess) return PP_OK;
  return e == cudaErrorMemoryAllocation ? PP_ENOMEM : PP_ECUDA;
}

// Device and pinned buffers of one call; released by the destructor.  Device
// buffers come from the stream-ordered allocator, whose default pool keeps
// freed memory for the next call.
struct Buffers {
  cudaStream_t cs = nullptr, hs = nullptr, ds = nullptr;  // compute, host->device, device->host
  cudaEvent_t ev_h2d[2] = {}, ev_d2d[2] = {}, ev_d2h[2] = {}, ev_info[2] = {};
  uint8_t* din[2] = {};
  uint8_t* stage[2] = {};
  void* scratch = nullptr;
  ChunkInfo* d_info[2] = {};
  ChunkInfo* h_info = nullptr;
  int32_t* d_off[2][MAX_STR_COLS] = {};
  uint8_t* d_chars[2][MAX_STR_COLS] = {};
  void* d_typed[2][PP_MAX_COLS] = {};
  cudaError_t alloc(void** p, size_t bytes) { return cudaMallocAsync(p, bytes, cs); }
  template <class T>
  void release(T* p) {
    if (p) cudaFreeAsync(p, cs);
  }
  ~Buffers() {
    if (hs) cudaStreamSynchronize(hs);
    if (ds) cudaStreamSynchronize(ds);
    for (int k = 0; k < 2; ++k) {
      release(din[k]);
      release(stage[k]);
      release(d_info[k]);
      for (int c = 0; c < MAX_STR_COLS; ++c) { release(d_off[k][c]); release(d_chars[k][c]); }
      for (int c = 0; c < PP_MAX_COLS; ++c) release(d_typed[k][c]);
      cudaEvent_t* evs[4] = {ev_h2d, ev_d2d, ev_d2h, ev_info};
      for (cudaEvent_t* ev : evs)
        if (ev[k]) cudaEventDestroy(ev[k]);
    }
    release(scratch);
    cudaStreamSynchronize(cs);
    if (h_info) cudaFreeHost(h_info);
    if (hs) cudaStreamDestroy(hs);
    if (ds) cudaStreamDestroy(ds);
  }
};

// Keep freed stream-ordered memory in the device's default pool across
// calls (the pool otherwise returns it to the system at every synchronize).
cudaError_t keep_pool_memory() {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaMemPool_t pool;
  if ((e = cudaDeviceGetDefaultMemPool(&pool, dev)) != cudaSuccess) return e;
  uint64_t keep = ~0ull;
  return cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
}

}  // namespace

extern "C" pp_rc pp_parse_host(const uint8_t* h_in, size_t n_bytes, const pp_dfa_desc* dfa,
                               int n_cols, const pp_coltype* col_types,
                               int32_t* const h_offsets[], uint8_t* const h_chars[],
                               void* const h_typed[], size_t records_capacity,
                               const size_t chars_capacity[], pp_status* h_status,
                               size_t chunk_bytes, cudaStream_t stream) {
  // the arguments are checked as pp_parse checks them (host pointers stand
  // in for the device ones)
  ppi::ParseParams p0;
  pp_rc rc = ppi::parse_prepare(h_in, n_bytes, dfa, n_cols, col_types, h_offsets, h_chars, h_typed,
                                records_capacity, chars_capacity, h_status, &p0);
  if (rc != PP_OK) return rc;
  const size_t tile = ppi::parse_tile_bytes();
  size_t chunk = chunk_bytes ? chunk_bytes : (size_t(128) << 20);
  chunk = std::max(tile, (chunk + tile - 1) / tile * tile);
  const size_t max_carry = chunk;       // a record may span at most one chunk's bytes
  const size_t in_cap = chunk + max_carry;
  const int n_str = p0.n_str;
  const int ns = ppi::parse_ns_width(n_str);
  const bool out = p0.has_out != 0;
  const size_t rec_cap = std::min<size_t>(records_capacity, in_cap) + 1;  // + the unfinished record
  size_t chars_cap[PP_MAX_COLS] = {};
  for (int c = 0; c < n_cols; ++c)
    if (out && col_types[c] == PP_COL_STRING) chars_cap[c] = std::min<size_t>(chars_capacity[c], in_cap);

  Buffers B;
  B.cs = stream;
  cudaError_t e = keep_pool_memory();
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&B.hs, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&B.ds, cudaStreamNonBlocking);
  for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
    if ((e = cudaEventCreateWithFlags(&B.ev_h2d[k], cudaEventDisableTiming)) != cudaSuccess) break;
    if ((e = cudaEventCreateWithFlags(&B.ev_d2d[k], cudaEventDisableTiming)) != cudaSuccess) break;
    if ((e = cudaEventCreateWithFlags(&B.ev_d2h[k], cudaEventDisableTiming)) != cudaSuccess) break;
    if ((e = cudaEventCreateWithFlags(&B.ev_info[k], cudaEventDisableTiming)) != cudaSuccess) break;
    if ((e = B.alloc(reinterpret_cast<void**>(&B.din[k]), in_cap + 16)) != cudaSuccess) break;
    if ((e = B.alloc(reinterpret_cast<void**>(&B.stage[k]), chunk)) != cudaSuccess) break;
    if ((e = B.alloc(reinterpret_cast<void**>(&B.d_info[k]), sizeof(ChunkInfo))) != cudaSuccess) break;
    if (!out) continue;
    for (int c = 0; c < n_cols && e == cudaSuccess; ++c) {
      const int ty = col_types[c];
      if (ty == PP_COL_STRING) {
        const int si = p0.stridx[c];
        if ((e = B.alloc(reinterpret_cast<void**>(&B.d_off[k][si]), (rec_cap + 1) * sizeof(int32_t))) != cudaSuccess) break;
        e = B.alloc(reinterpret_cast<void**>(&B.d_chars[k][si]), std::max<size_t>(chars_cap[c], 1));
      } else if (ty != PP_COL_SKIP) {
        e = B.alloc(&B.d_typed[k][c], rec_cap * width_of(ty));
      }
    }
  }
  if (e == cudaSuccess)
    e = B.alloc(&B.scratch, ppi::parse_scratch_bytes(uint32_t((in_cap + tile - 1) / tile), ns, n_cols));
  if (e == cudaSuccess) e = cudaMallocHost(&B.h_info, 2 * sizeof(ChunkInfo));
  if (e != cudaSuccess) return rc_of(e);

  // per-chunk output pointer tables, by column (as pp_parse takes them)
  int32_t* off_c[2][PP_MAX_COLS] = {};
  uint8_t* chars_c[2][PP_MAX_COLS] = {};
  for (int k = 0; k < 2; ++k)
    for (int c = 0; c < n_cols; ++c)
      if (out && col_types[c] == PP_COL_STRING) {
        off_c[k][c] = B.d_off[k][p0.stridx[c]];
        chars_c[k][c] = B.d_chars[k][p0.stridx[c]];
      }

  int32_t merged_err = 0;
  uint64_t first_err = ~0ull;
  uint64_t rec_base = 0;
  uint64_t chars_base[MAX_STR_COLS] = {};
  size_t pos = 0, carry = 0;
  const uint8_t* carry_src = nullptr;
  if (n_bytes) {
    const size_t l0 = std::min(chunk, n_bytes);
    if ((e = cudaMemcpyAsync(B.stage[0], h_in, l0, cudaMemcpyHostToDevice, B.hs)) != cudaSuccess ||
        (e = cudaEventRecord(B.ev_h2d[0], B.hs)) != cudaSuccess)
      return rc_of(e);
  }
  for (int i = 0;; ++i) {
    const int k = i & 1;
    const size_t nl = std::min(chunk, n_bytes - pos);  // new bytes of this chunk
    const bool last = pos + nl == n_bytes;
    if (!last) {  // the next chunk's new bytes, once its staging buffer is free
      const size_t nn = std::min(chunk, n_bytes - pos - nl);
      if ((e = cudaStreamWaitEvent(B.hs, B.ev_d2d[k ^ 1], 0)) != cudaSuccess ||
          (e = cudaMemcpyAsync(B.stage[k ^ 1], h_in + pos + nl, nn, cudaMemcpyHostToDevice, B.hs)) !=
              cudaSuccess ||
          (e = cudaEventRecord(B.ev_h2d[k ^ 1], B.hs)) != cudaSuccess)
        return rc_of(e);
    }
    // this chunk's input: the carried bytes, then the staged ones
    if ((e = cudaStreamWaitEvent(B.cs, B.ev_h2d[k], 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(B.cs, B.ev_d2h[k], 0)) != cudaSuccess)
      return rc_of(e);
    if (carry && (e = cudaMemcpyAsync(B.din[k], carry_src, carry, cudaMemcpyDeviceToDevice, B.cs)) !=
                     cudaSuccess)
      return rc_of(e);
    if (nl && (e = cudaMemcpyAsync(B.din[k] + carry, B.stage[k], nl, cudaMemcpyDeviceToDevice, B.cs)) !=
                  cudaSuccess)
      return rc_of(e);
    if ((e = cudaEventRecord(B.ev_d2d[k], B.cs)) != cudaSuccess) return rc_of(e);
    const size_t len = carry + nl;

    ppi::ParseParams p;
    rc = ppi::parse_prepare(B.din[k], len, dfa, n_cols, col_types, out ? off_c[k] : nullptr,
                            out ? chars_c[k] : nullptr, out ? B.d_typed[k] : nullptr, rec_cap,
                            chars_cap, &B.d_info[k]->st, &p);
    if (rc != PP_OK) return rc;
    if ((e = cudaMemsetAsync(B.d_info[k], 0, sizeof(ChunkInfo), B.cs)) != cudaSuccess) return rc_of(e);
    p.record_end = last ? nullptr : &B.d_info[k]->record_end;
    ppi::parse_scratch_carve(B.scratch, p.n_tiles, ns, n_cols, &p.s);
    if ((e = ppi::launch_parse(p, B.cs)) != cudaSuccess) return rc_of(e);
    if (out && n_str) {
      RebaseArgs a{};
      for (int si = 0; si < n_str; ++si) {
        a.off[si] = B.d_off[k][si];
        a.base[si] = int64_t(chars_base[si]);
      }
      a.n_str = n_str;
      a.ci = B.d_info[k];
      rebase_kernel<<<256, 256, 0, B.cs>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return rc_of(e);
    }
    if ((e = cudaMemcpyAsync(&B.h_info[k], B.d_info[k], sizeof(ChunkInfo), cudaMemcpyDeviceToHost,
                             B.cs)) != cudaSuccess ||
        (e = cudaEventRecord(B.ev_info[k], B.cs)) != cudaSuccess ||
        (e = cudaEventSynchronize(B.ev_info[k])) != cudaSuccess)
      return rc_of(e);

    // merge the chunk's summary
    const ChunkInfo& ci = B.h_info[k];
    const uint64_t g0 = pos - carry;  // input offset of the chunk's first byte
    merged_err |= ci.st.error;
    if (ci.st.first_error_offset != ~0ull) first_err = std::min(first_err, g0 + ci.st.first_error_offset);
    uint64_t nrec = ci.st.n_records;
    bool fits = rec_base + nrec <= records_capacity || !out;
    for (int si = 0; si < n_str && out; ++si) {
      const int c = p.strcol[si];
      if (chars_base[si] + ci.chars[si] > chars_capacity[c] ||
          chars_base[si] + ci.chars[si] > 0x7FFFFFFFull)
        fits = false;
    }
    if (!fits) {
      merged_err |= PP_ERR_CAPACITY;
      break;
    }
    // After a fatal error the outputs are undefined (as for pp_parse) and the
    // invalid state would hold every later byte: stop here.
    if (merged_err & PP_ERR_FATAL) break;
    // the chunk's complete records -> host
    if (out && nrec) {
      if ((e = cudaStreamWaitEvent(B.ds, B.ev_info[k], 0)) != cudaSuccess) return rc_of(e);
      for (int c = 0; c < n_cols && e == cudaSuccess; ++c) {
        const int ty = col_types[c];
        if (ty == PP_COL_STRING) {
          const int si = p0.stridx[c];
          e = cudaMemcpyAsync(h_offsets[c] + rec_base + 1, B.d_off[k][si] + 1, nrec * sizeof(int32_t),
                              cudaMemcpyDeviceToHost, B.ds);
          if (e == cudaSuccess && ci.chars[si])
            e = cudaMemcpyAsync(h_chars[c] + chars_base[si], B.d_chars[k][si], ci.chars[si],
                                cudaMemcpyDeviceToHost, B.ds);
        } else if (ty != PP_COL_SKIP && h_typed[c]) {
          const size_t w = width_of(ty);
          e = cudaMemcpyAsync(static_cast<uint8_t*>(h_typed[c]) + rec_base * w, B.d_typed[k][c],
                              nrec * w, cudaMemcpyDeviceToHost, B.ds);
        }
      }
      if (e != cudaSuccess) return rc_of(e);
    }
    if ((e = cudaEventRecord(B.ev_d2h[k], B.ds)) != cudaSuccess) return rc_of(e);
    rec_base += nrec;
    for (int si = 0; si < n_str; ++si) chars_base[si] += ci.chars[si];
    if (last) break;
    // the unfinished record moves to the front of the next chunk
    const uint64_t re = ci.record_end;
    carry = len - re;
    carry_src = B.din[k] + re;
    pos += nl;
    if (carry > max_carry) {
      merged_err |= PP_ERR_CAPACITY;
      if (first_err == ~0ull) first_err = g0 + re;
      cudaStreamSynchronize(B.ds);
      std::memset(h_status, 0, sizeof *h_status);
      h_status->error = merged_err;
      h_status->first_error_offset = first_err;
      h_status->n_records = rec_base;
      return PP_ECHUNK;
    }
  }
  if ((e = cudaStreamSynchronize(B.ds)) != cudaSuccess) return rc_of(e);
  std::memset(h_status, 0, sizeof *h_status);
  h_status->error = merged_err;
  h_status->first_error_offset = first_err;
  h_status->n_records = rec_base;
  for (int si = 0; si < n_str; ++si) {
    const int c = p0.strcol[si];
    h_status->chars_len[c] = chars_base[si];
    if (out) h_offsets[c][0] = 0;
  }
  return PP_OK;
}
