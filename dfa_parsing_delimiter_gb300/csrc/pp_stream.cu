// pp_parse_host and pp_tokenize_host: an input in host memory into outputs
// in host memory, streamed through the device in chunks so that the copies
// in both directions overlap the device work (ParPaRaw Section 4, the
// streaming set-up: the input moves to the device in partitions while
// earlier partitions are parsed and their results move back).
//
// Per chunk i, on the caller's stream (cs) unless noted:
//   h2d stream:   new bytes of chunk i+1, host -> device staging buffer
//   cs:           input i = bytes carried over from chunk i-1 ++ staged bytes;
//                 the device pass in partial mode (all but the last chunk):
//                 the record (token) still open at the chunk end is left
//                 open, and where it starts is reported;
//                 outputs rebased to whole-input positions;
//                 chunk summary -> host
//   host:         waits for the summary, merges the status, and carries the
//                 open record (token) to the front of chunk i+1's input
//   d2h stream:   chunk i's complete records (tokens), device -> host outputs
// Two sets of device buffers alternate between chunks; the two copy
// directions run on streams of their own, so both copy engines work at once.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_internal.h"

namespace {

using ppi::MAX_STR_COLS;

pp_rc rc_of(cudaError_t e) {
  if (e == cudaSuccess) return PP_OK;
  return e == cudaErrorMemoryAllocation ? PP_ENOMEM : PP_ECUDA;
}

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

size_t round_chunk(size_t chunk_bytes) {
  const size_t tile = ppi::parse_tile_bytes();
  const size_t c = chunk_bytes ? chunk_bytes : (size_t(128) << 20);
  return std::max(tile, (c + tile - 1) / tile * tile);
}

// Streams, events, the input buffers and the chunk summaries of one call.
// Device memory comes from the stream-ordered allocator and is released,
// with the rest, by the destructor.
struct Pipeline {
  cudaStream_t cs = nullptr, hs = nullptr, ds = nullptr;  // device work, host->device, device->host
  cudaEvent_t ev_h2d[2] = {}, ev_d2d[2] = {}, ev_d2h[2] = {}, ev_info[2] = {};
  uint8_t* din[2] = {};    // chunk input: carry ++ new bytes
  uint8_t* stage[2] = {};  // new bytes as copied from the host
  void* d_info[2] = {};    // chunk summary (device) ...
  uint8_t* h_info = nullptr;  // ... and its pinned host copy, 2 x info_bytes
  size_t info_bytes = 0;
  std::vector<void*> owned;

  cudaError_t alloc(void** p, size_t bytes) {
    const cudaError_t e = cudaMallocAsync(p, std::max<size_t>(bytes, 1), cs);
    if (e == cudaSuccess) owned.push_back(*p);
    return e;
  }
  cudaError_t init(cudaStream_t stream, size_t chunk, size_t in_cap, size_t info) {
    cs = stream;
    info_bytes = info;
    cudaError_t e = keep_pool_memory();
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ds, cudaStreamNonBlocking);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
      cudaEvent_t* evs[4] = {&ev_h2d[k], &ev_d2d[k], &ev_d2h[k], &ev_info[k]};
      for (cudaEvent_t* ev : evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
      if (e == cudaSuccess) e = alloc(reinterpret_cast<void**>(&din[k]), in_cap + 16);
      if (e == cudaSuccess) e = alloc(reinterpret_cast<void**>(&stage[k]), chunk);
      if (e == cudaSuccess) e = alloc(&d_info[k], info);
    }
    if (e == cudaSuccess) e = cudaMallocHost(&h_info, 2 * info);
    return e;
  }
  // new bytes of a chunk into staging buffer k, once chunk k's input copy
  // no longer needs it
  cudaError_t h2d(int k, const uint8_t* src, size_t n) {
    cudaError_t e = cudaStreamWaitEvent(hs, ev_d2d[k], 0);
    if (e == cudaSuccess && n) e = cudaMemcpyAsync(stage[k], src, n, cudaMemcpyHostToDevice, hs);
    if (e == cudaSuccess) e = cudaEventRecord(ev_h2d[k], hs);
    return e;
  }
  // input buffer k = carry ++ staged bytes, once buffer set k's earlier
  // results have reached the host
  cudaError_t assemble(int k, const uint8_t* carry_src, size_t carry, size_t nl) {
    cudaError_t e = cudaStreamWaitEvent(cs, ev_h2d[k], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev_d2h[k], 0);
    if (e == cudaSuccess && carry)
      e = cudaMemcpyAsync(din[k], carry_src, carry, cudaMemcpyDeviceToDevice, cs);
    if (e == cudaSuccess && nl)
      e = cudaMemcpyAsync(din[k] + carry, stage[k], nl, cudaMemcpyDeviceToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev_d2d[k], cs);
    return e;
  }
  // chunk summary k -> host (waits)
  cudaError_t summary(int k) {
    cudaError_t e = cudaMemcpyAsync(h_info + k * info_bytes, d_info[k], info_bytes,
                                    cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev_info[k], cs);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev_info[k]);
    return e;
  }
  cudaError_t d2h_begin(int k) { return cudaStreamWaitEvent(ds, ev_info[k], 0); }
  cudaError_t d2h(void* dst, const void* src, size_t n) {
    return n ? cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, ds) : cudaSuccess;
  }
  cudaError_t d2h_end(int k) { return cudaEventRecord(ev_d2h[k], ds); }

  ~Pipeline() {
    if (hs) cudaStreamSynchronize(hs);
    if (ds) cudaStreamSynchronize(ds);
    for (void* p : owned) cudaFreeAsync(p, cs);
    cudaStreamSynchronize(cs);
    for (int k = 0; k < 2; ++k) {
      cudaEvent_t evs[4] = {ev_h2d[k], ev_d2d[k], ev_d2h[k], ev_info[k]};
      for (cudaEvent_t ev : evs)
        if (ev) cudaEventDestroy(ev);
    }
    if (h_info) cudaFreeHost(h_info);
    if (hs) cudaStreamDestroy(hs);
    if (ds) cudaStreamDestroy(ds);
  }
};

void finish_status(pp_status* h, int32_t err, uint64_t first, uint64_t records, uint64_t tokens) {
  std::memset(h, 0, sizeof *h);
  h->error = err;
  h->first_error_offset = first;
  h->n_records = records;
  h->n_tokens = tokens;
}

// ------------------------------------------------------------ records
// Device summary of one parse chunk.
struct ParseInfo {
  pp_status st;
  unsigned long long record_end;   // 1 + the chunk's last record delimiter (0: none)
  uint64_t chars[MAX_STR_COLS];    // chars of the chunk's complete records per string column
};

struct RebaseArgs {
  int32_t* off[MAX_STR_COLS];
  int64_t base[MAX_STR_COLS];
  int n_str;
  ParseInfo* ci;
};

// Records the chars of the chunk's complete records (offsets[n_records])
// and adds the chars emitted by earlier chunks to offsets[1..n_records].
// The host has checked that the sums fit in int32.
__global__ void rebase_offsets_kernel(RebaseArgs a) {
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
    case PP_COL_INT64: case PP_COL_FLOAT64: case PP_COL_TIMESTAMP: return 8;
    default: return 0;
  }
}

// ------------------------------------------------------------ tokens
// Device summary of one token chunk: status, then (partial mode) 1 + the
// last token start and the DFA state before it.
struct TokInfo {
  pp_status st;
  unsigned long long carry[2];
};

// starts of the chunk's complete tokens: chunk-relative -> input positions
__global__ void rebase_starts_kernel(uint64_t* start, const TokInfo* ti, uint64_t base, bool last) {
  const uint64_t t = ti->st.n_tokens;
  const uint64_t n = last ? t : (t ? t - 1 : 0);
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += uint64_t(gridDim.x) * blockDim.x)
    start[i] += base;
}

}  // namespace

extern "C" {

pp_rc pp_parse_host(const uint8_t* h_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                    const pp_coltype* col_types, int32_t* const h_offsets[],
                    uint8_t* const h_chars[], void* const h_typed[], size_t records_capacity,
                    const size_t chars_capacity[], pp_status* h_status, size_t chunk_bytes,
                    cudaStream_t stream) {
  // the arguments are checked as pp_parse checks them (host pointers stand
  // in for the device ones); inputs in a multi-byte encoding are not
  // streamed (a chunk could end inside a symbol)
  if (dfa && dfa->encoding != PP_ENC_BYTES) return PP_EINVAL;
  ppi::ParseParams p0;
  pp_rc rc = ppi::parse_prepare(h_in, n_bytes, dfa, n_cols, col_types, h_offsets, h_chars, h_typed,
                                records_capacity, chars_capacity, h_status, &p0);
  if (rc != PP_OK) return rc;
  const size_t tile = ppi::parse_tile_bytes();
  const size_t chunk = round_chunk(chunk_bytes);
  const size_t max_carry = chunk;  // a record may span at most one chunk's bytes
  const size_t in_cap = chunk + max_carry;
  const int n_str = p0.n_str;
  const int ns = ppi::parse_ns_width(n_str);
  const bool out = p0.has_out != 0;
  const size_t rec_cap = std::min<size_t>(records_capacity, in_cap) + 1;  // + the open record
  size_t chars_cap[PP_MAX_COLS] = {};
  for (int c = 0; c < n_cols; ++c)
    if (out && col_types[c] == PP_COL_STRING) chars_cap[c] = std::min<size_t>(chars_capacity[c], in_cap);

  Pipeline B;
  cudaError_t e = B.init(stream, chunk, in_cap, sizeof(ParseInfo));
  // per buffer set, outputs by column (as pp_parse takes them)
  int32_t* off_c[2][PP_MAX_COLS] = {};
  uint8_t* chars_c[2][PP_MAX_COLS] = {};
  void* typed_c[2][PP_MAX_COLS] = {};
  for (int k = 0; k < 2 && out; ++k)
    for (int c = 0; c < n_cols && e == cudaSuccess; ++c) {
      const int ty = col_types[c];
      if (ty == PP_COL_STRING) {
        e = B.alloc(reinterpret_cast<void**>(&off_c[k][c]), (rec_cap + 1) * sizeof(int32_t));
        if (e == cudaSuccess) e = B.alloc(reinterpret_cast<void**>(&chars_c[k][c]), chars_cap[c]);
      } else if (ty != PP_COL_SKIP) {
        e = B.alloc(&typed_c[k][c], rec_cap * width_of(ty));
      }
    }
  void* scratch = nullptr;
  if (e == cudaSuccess)
    e = B.alloc(&scratch, ppi::parse_scratch_bytes(uint32_t((in_cap + tile - 1) / tile), ns));
  if (e != cudaSuccess) return rc_of(e);

  int32_t merged_err = 0;
  uint64_t first_err = ~0ull, rec_base = 0;
  uint64_t chars_base[MAX_STR_COLS] = {};
  size_t pos = 0, carry = 0;
  const uint8_t* carry_src = nullptr;
  if ((e = B.h2d(0, h_in, std::min(chunk, n_bytes))) != cudaSuccess) return rc_of(e);
  for (int i = 0;; ++i) {
    const int k = i & 1;
    const size_t nl = std::min(chunk, n_bytes - pos);  // new bytes of this chunk
    const bool last = pos + nl == n_bytes;
    if (!last && (e = B.h2d(k ^ 1, h_in + pos + nl, std::min(chunk, n_bytes - pos - nl))) != cudaSuccess)
      return rc_of(e);
    if ((e = B.assemble(k, carry_src, carry, nl)) != cudaSuccess) return rc_of(e);
    const size_t len = carry + nl;
    ParseInfo* di = static_cast<ParseInfo*>(B.d_info[k]);
    ppi::ParseParams p;
    rc = ppi::parse_prepare(B.din[k], len, dfa, n_cols, col_types, out ? off_c[k] : nullptr,
                            out ? chars_c[k] : nullptr, out ? typed_c[k] : nullptr, rec_cap,
                            chars_cap, &di->st, &p);
    if (rc != PP_OK) return rc;
    if ((e = cudaMemsetAsync(di, 0, sizeof(ParseInfo), B.cs)) != cudaSuccess) return rc_of(e);
    p.record_end = last ? nullptr : &di->record_end;
    ppi::parse_scratch_carve(scratch, p.n_tiles, ns, &p.s);
    if ((e = ppi::launch_parse(p, B.cs)) != cudaSuccess) return rc_of(e);
    if (out && n_str) {
      RebaseArgs a{};
      for (int si = 0; si < n_str; ++si) {
        a.off[si] = p.offsets[si];
        a.base[si] = int64_t(chars_base[si]);
      }
      a.n_str = n_str;
      a.ci = di;
      rebase_offsets_kernel<<<256, 256, 0, B.cs>>>(a);
      if ((e = cudaGetLastError()) != cudaSuccess) return rc_of(e);
    }
    if ((e = B.summary(k)) != cudaSuccess) return rc_of(e);

    // merge the chunk's summary
    const ParseInfo& ci = *reinterpret_cast<const ParseInfo*>(B.h_info + k * sizeof(ParseInfo));
    const uint64_t g0 = pos - carry;  // input offset of the chunk's first byte
    merged_err |= ci.st.error;
    if (ci.st.first_error_offset != ~0ull) first_err = std::min(first_err, g0 + ci.st.first_error_offset);
    const uint64_t nrec = ci.st.n_records;
    bool fits = rec_base + nrec <= records_capacity || !out;
    for (int si = 0; si < n_str && out; ++si) {
      const uint64_t end = chars_base[si] + ci.chars[si];
      if (end > chars_capacity[p.strcol[si]] || end > 0x7FFFFFFFull) fits = false;
    }
    if (!fits) {
      merged_err |= PP_ERR_CAPACITY;
      break;
    }
    // After a fatal error the outputs are undefined (as for pp_parse) and
    // the invalid state would hold every later byte: stop here.
    if (merged_err & PP_ERR_FATAL) break;
    // the chunk's complete records -> host
    if (out && nrec) {
      if ((e = B.d2h_begin(k)) != cudaSuccess) return rc_of(e);
      for (int c = 0; c < n_cols && e == cudaSuccess; ++c) {
        const int ty = col_types[c];
        if (ty == PP_COL_STRING) {
          const int si = p0.stridx[c];
          e = B.d2h(h_offsets[c] + rec_base + 1, off_c[k][c] + 1, nrec * sizeof(int32_t));
          if (e == cudaSuccess) e = B.d2h(h_chars[c] + chars_base[si], chars_c[k][c], ci.chars[si]);
        } else if (ty != PP_COL_SKIP && h_typed[c]) {
          const size_t w = width_of(ty);
          e = B.d2h(static_cast<uint8_t*>(h_typed[c]) + rec_base * w, typed_c[k][c], nrec * w);
        }
      }
      if (e != cudaSuccess) return rc_of(e);
    }
    if ((e = B.d2h_end(k)) != cudaSuccess) return rc_of(e);
    rec_base += nrec;
    for (int si = 0; si < n_str; ++si) chars_base[si] += ci.chars[si];
    if (last) break;
    // the open record moves to the front of the next chunk
    const uint64_t re = ci.record_end;
    carry = len - re;
    carry_src = B.din[k] + re;
    pos += nl;
    if (carry > max_carry) {
      cudaStreamSynchronize(B.ds);
      finish_status(h_status, merged_err | PP_ERR_CAPACITY,
                    first_err == ~0ull ? g0 + re : first_err, rec_base, 0);
      return PP_ECHUNK;
    }
  }
  if ((e = cudaStreamSynchronize(B.ds)) != cudaSuccess) return rc_of(e);
  finish_status(h_status, merged_err, first_err, rec_base, 0);
  for (int si = 0; si < n_str; ++si) {
    const int c = p0.strcol[si];
    h_status->chars_len[c] = chars_base[si];
    if (out) h_offsets[c][0] = 0;
  }
  return PP_OK;
}

pp_rc pp_tokenize_host(const uint8_t* h_in, size_t n_bytes, const pp_dfa_desc* dfa,
                       uint8_t* h_token_id, uint64_t* h_start, uint32_t* h_len,
                       size_t tokens_capacity, pp_status* h_status, size_t chunk_bytes,
                       cudaStream_t stream) {
  if (!h_status || (n_bytes && !h_in) || !ppi::generic_dfa_ok(dfa)) return PP_EINVAL;
  if (tokens_capacity && (!h_token_id || !h_start || !h_len)) return PP_EINVAL;
  const bool out = tokens_capacity > 0;
  const size_t chunk = round_chunk(chunk_bytes);
  const size_t max_carry = chunk;  // a token may span at most one chunk's bytes
  const size_t in_cap = chunk + max_carry;
  const size_t tok_cap = out ? std::min<size_t>(tokens_capacity, in_cap) + 1 : 0;
  ppi::GenericDfa g = ppi::to_generic_dfa(dfa);

  Pipeline B;
  cudaError_t e = B.init(stream, chunk, in_cap, sizeof(TokInfo));
  uint8_t* d_id[2] = {};
  uint64_t* d_start[2] = {};
  uint32_t* d_len[2] = {};
  for (int k = 0; k < 2 && out && e == cudaSuccess; ++k) {
    e = B.alloc(reinterpret_cast<void**>(&d_id[k]), tok_cap);
    if (e == cudaSuccess) e = B.alloc(reinterpret_cast<void**>(&d_start[k]), tok_cap * 8);
    if (e == cudaSuccess) e = B.alloc(reinterpret_cast<void**>(&d_len[k]), tok_cap * 4);
  }
  void* scratch = nullptr;
  const size_t sb = ppi::tokenize_scratch_bytes(in_cap);
  if (e == cudaSuccess) e = B.alloc(&scratch, sb);
  if (e != cudaSuccess) return rc_of(e);

  int32_t merged_err = 0;
  uint64_t first_err = ~0ull, tok_base = 0;
  size_t pos = 0, carry = 0;
  const uint8_t* carry_src = nullptr;
  if ((e = B.h2d(0, h_in, std::min(chunk, n_bytes))) != cudaSuccess) return rc_of(e);
  for (int i = 0;; ++i) {
    const int k = i & 1;
    const size_t nl = std::min(chunk, n_bytes - pos);
    const bool last = pos + nl == n_bytes;
    if (!last && (e = B.h2d(k ^ 1, h_in + pos + nl, std::min(chunk, n_bytes - pos - nl))) != cudaSuccess)
      return rc_of(e);
    if ((e = B.assemble(k, carry_src, carry, nl)) != cudaSuccess) return rc_of(e);
    const size_t len = carry + nl;
    const uint64_t g0 = pos - carry;
    TokInfo* di = static_cast<TokInfo*>(B.d_info[k]);
    if ((e = cudaMemsetAsync(di, 0, sizeof(TokInfo), B.cs)) != cudaSuccess) return rc_of(e);
    if ((e = ppi::launch_tokenize(B.din[k], len, g, d_id[k], d_start[k], d_len[k], tok_cap, &di->st,
                                  scratch, sb, B.cs, last ? nullptr : di->carry)) != cudaSuccess)
      return rc_of(e);
    if (out && g0) {
      rebase_starts_kernel<<<256, 256, 0, B.cs>>>(d_start[k], di, g0, last);
      if ((e = cudaGetLastError()) != cudaSuccess) return rc_of(e);
    }
    if ((e = B.summary(k)) != cudaSuccess) return rc_of(e);

    const TokInfo& ci = *reinterpret_cast<const TokInfo*>(B.h_info + k * sizeof(TokInfo));
    merged_err |= ci.st.error;
    if (ci.st.first_error_offset != ~0ull) first_err = std::min(first_err, g0 + ci.st.first_error_offset);
    const uint64_t t = ci.st.n_tokens;
    const uint64_t ntok = last ? t : (t ? t - 1 : 0);  // the open token goes on in the next chunk
    if (out && tok_base + ntok > tokens_capacity) {
      merged_err |= PP_ERR_CAPACITY;
      break;
    }
    if (merged_err & PP_ERR_FATAL) break;
    if (out && ntok) {
      if ((e = B.d2h_begin(k)) != cudaSuccess ||
          (e = B.d2h(h_token_id + tok_base, d_id[k], ntok)) != cudaSuccess ||
          (e = B.d2h(h_start + tok_base, d_start[k], ntok * 8)) != cudaSuccess ||
          (e = B.d2h(h_len + tok_base, d_len[k], ntok * 4)) != cudaSuccess)
        return rc_of(e);
    }
    if ((e = B.d2h_end(k)) != cudaSuccess) return rc_of(e);
    tok_base += ntok;
    if (last) break;
    // the open token, from its start, moves to the front of the next
    // chunk, which starts in the DFA state the token started from
    const uint64_t ls = ci.carry[0] ? ci.carry[0] - 1 : 0;
    carry = len - ls;
    carry_src = B.din[k] + ls;
    g.start_state = uint8_t(ci.carry[1]);
    pos += nl;
    if (carry > max_carry) {
      cudaStreamSynchronize(B.ds);
      finish_status(h_status, merged_err | PP_ERR_CAPACITY,
                    first_err == ~0ull ? g0 + ls : first_err, 0, tok_base);
      return PP_ECHUNK;
    }
  }
  if ((e = cudaStreamSynchronize(B.ds)) != cudaSuccess) return rc_of(e);
  finish_status(h_status, merged_err, first_err, 0, tok_base);
  return PP_OK;
}

}  // extern "C"
