// pp_parse_ex: pp_parse with the parse options of ParPaRaw Section 4.
//
//  * Column defaults ("Default values for empty strings"): the tile pass
//    stores the column's default for an empty or missing numeric field.
//  * Skipping rows ("Skipping rows"): rows are lines, cut at every
//    record-delimiter byte whatever the quoting, and they must go before the
//    DFA runs; an initial parallel pass compacts the input without them:
//    record-delimiter counts per block, their exclusive scan, the byte range
//    of each skipped row (a search in that scan, then in the block), the
//    ranges' prefix sums, and a copy that drops the ranges.
//  * Skipping records and rejecting records with the wrong field count
//    ("Skipping records and selecting columns", "Inferring or validating
//    number of columns"): a bitmap over the input's records marks the ones
//    not to emit (the skip list scattered into it; with rejection, a status
//    pass of the tile kernel adds every record whose field count is not the
//    schema's), its per-group prefix sums give each emitted record its
//    output row, and the tile pass then writes only emitted records.
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>

#include "pp.h"
#include "pp_internal.h"

namespace {

constexpr uint32_t RB = 4096;   // bytes per block of the row count
constexpr int SCAN_T = 1024;    // one-block scans

// record-delimiter bytes per RB-byte block
__global__ void row_count_kernel(const uint8_t* in, uint64_t n, uint8_t rd, uint32_t* cnt,
                                 uint64_t nb) {
  for (uint64_t blk = blockIdx.x; blk < nb; blk += gridDim.x) {
    const uint64_t b0 = blk * RB, b1 = min(n, b0 + RB);
    uint32_t c = 0;
    for (uint64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) c += in[i] == rd ? 1u : 0u;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    __shared__ uint32_t ws[8];
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t s = 0;
      for (int w = 0; w < int(blockDim.x / 32); ++w) s += ws[w];
      cnt[blk] = s;
    }
    __syncthreads();
  }
}

// out[i] = sum of in[0..i) (one block; from in64 or else in32), out[n] = total
__global__ void exclusive_scan_kernel(const uint64_t* in64, const uint32_t* in32, uint64_t n,
                                      uint64_t* out) {
  __shared__ uint64_t part[SCAN_T];
  const uint64_t per = (n + SCAN_T - 1) / SCAN_T;
  const uint64_t i0 = min(n, uint64_t(threadIdx.x) * per), i1 = min(n, i0 + per);
  uint64_t s = 0;
  for (uint64_t i = i0; i < i1; ++i) s += in64 ? in64[i] : in32[i];
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t run = 0;
    for (int k = 0; k < SCAN_T; ++k) {
      const uint64_t v = part[k];
      part[k] = run;
      run += v;
    }
    out[n] = run;
  }
  __syncthreads();
  uint64_t run = part[threadIdx.x];
  for (uint64_t i = i0; i < i1; ++i) {
    const uint64_t v = in64 ? in64[i] : in32[i];
    out[i] = run;
    run += v;
  }
}

// position + 1 of the k-th (0-based) record-delimiter byte, or n when there
// are not that many
__device__ uint64_t rd_end(const uint8_t* in, uint64_t n, uint8_t rd, const uint64_t* rows_before,
                           uint64_t nb, uint64_t k) {
  if (k >= rows_before[nb]) return n;
  uint64_t lo = 0, hi = nb;  // the last block with rows_before <= k
  while (hi - lo > 1) {
    const uint64_t mid = (lo + hi) >> 1;
    if (rows_before[mid] <= k) lo = mid;
    else hi = mid;
  }
  uint64_t left = k - rows_before[lo];
  for (uint64_t i = lo * RB; i < n; ++i)
    if (in[i] == rd && left-- == 0) return i + 1;
  return n;
}

// byte range [start, end) of each skipped row
__global__ void row_range_kernel(const uint8_t* in, uint64_t n, uint8_t rd,
                                 const uint64_t* rows_before, uint64_t nb, const uint64_t* rows,
                                 uint64_t n_rows, uint64_t* rstart, uint64_t* rlen) {
  const uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_rows) return;
  const uint64_t r = rows[i];
  const uint64_t a = r == 0 ? 0ull : rd_end(in, n, rd, rows_before, nb, r - 1);
  const uint64_t b = rd_end(in, n, rd, rows_before, nb, r);
  rstart[i] = a;
  rlen[i] = b > a ? b - a : 0ull;
}

// copy the input without the ranges (sorted, disjoint); skipped[i] = bytes
// of the ranges before range i
__global__ void drop_ranges_kernel(const uint8_t* in, uint64_t n, const uint64_t* rstart,
                                   const uint64_t* rlen, const uint64_t* skipped, uint64_t n_rg,
                                   uint8_t* out) {
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x * 16;
  for (uint64_t p0 = (uint64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 16; p0 < n; p0 += stride) {
    // the first range that ends after p0
    uint64_t lo = 0, hi = n_rg;
    while (lo < hi) {
      const uint64_t mid = (lo + hi) >> 1;
      if (rstart[mid] + rlen[mid] <= p0) lo = mid + 1;
      else hi = mid;
    }
    uint64_t g = lo;
    const uint64_t p1 = min(n, p0 + 16);
    for (uint64_t p = p0; p < p1; ++p) {
      while (g < n_rg && rstart[g] + rlen[g] <= p) ++g;
      if (g < n_rg && p >= rstart[g]) continue;  // inside a skipped row
      out[p - skipped[g]] = in[p];
    }
  }
}

// set bit r for every listed record r < n_bits
__global__ void scatter_bits_kernel(const uint64_t* list, uint64_t n_list, uint64_t n_bits,
                                    uint32_t* bits) {
  const uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_list) return;
  const uint64_t r = list[i];
  if (r < n_bits) atomicOr(&bits[r >> 5], 1u << (r & 31u));
}

// bits set per group of 8 words
__global__ void group_count_kernel(const uint32_t* bits, uint64_t n_groups, uint64_t* cnt) {
  const uint64_t g = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  uint64_t c = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) c += __popc(bits[8 * g + k]);
  cnt[g] = c;
}

pp_rc rc_of(cudaError_t e) {
  if (e == cudaSuccess) return PP_OK;
  return e == cudaErrorMemoryAllocation ? PP_ENOMEM : PP_ECUDA;
}

bool ascending(const uint64_t* v, uint64_t n) {
  for (uint64_t i = 1; i < n; ++i)
    if (v[i] < v[i - 1]) return false;
  return true;
}

// the record-delimiter byte: the one byte the start state reads as a
// record delimiter (PP_EINVAL when there is not exactly one)
int rd_byte(const pp_dfa_desc* d) {
  int found = -1;
  for (int b = 0; b < 256; ++b)
    if (d->tag[d->start_state][d->byte_to_group[b]] == PP_TAG_RD) {
      if (found >= 0) return -1;
      found = b;
    }
  return found;
}

// Stream-ordered allocations released together.
struct Allocs {
  cudaStream_t s;
  std::vector<void*> v;
  explicit Allocs(cudaStream_t st) : s(st) {}
  cudaError_t get(void** p, size_t bytes) {
    const cudaError_t e = cudaMallocAsync(p, std::max<size_t>(bytes, 16), s);
    if (e == cudaSuccess) v.push_back(*p);
    return e;
  }
  ~Allocs() {
    for (void* p : v) cudaFreeAsync(p, s);
  }
};

}  // namespace

extern "C" pp_rc pp_parse_ex(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                             int n_cols, const pp_coltype* col_types, const pp_parse_opts* opts,
                             int32_t* const out_offsets[], uint8_t* const out_chars[],
                             void* const out_typed[], size_t records_capacity,
                             const size_t chars_capacity[], pp_status* d_status,
                             cudaStream_t stream) {
  pp_parse_opts o;
  std::memset(&o, 0, sizeof o);
  if (opts) o = *opts;
  if (o.flags & ~PP_PARSE_REJECT) return PP_EINVAL;
  // rows are cut at record-delimiter bytes: byte inputs only
  if (o.n_skip_rows && dfa && dfa->encoding != PP_ENC_BYTES) return PP_EINVAL;
  if ((o.n_skip_records && !o.skip_records) || (o.n_skip_rows && !o.skip_rows)) return PP_EINVAL;
  if (!ascending(o.skip_records, o.n_skip_records) || !ascending(o.skip_rows, o.n_skip_rows))
    return PP_EINVAL;
  // the lists without repeats
  std::vector<uint64_t> skip_rec(o.skip_records, o.skip_records + o.n_skip_records);
  std::vector<uint64_t> skip_row(o.skip_rows, o.skip_rows + o.n_skip_rows);
  skip_rec.erase(std::unique(skip_rec.begin(), skip_rec.end()), skip_rec.end());
  skip_row.erase(std::unique(skip_row.begin(), skip_row.end()), skip_row.end());
  o.skip_records = skip_rec.data();
  o.n_skip_records = skip_rec.size();
  o.skip_rows = skip_row.data();
  o.n_skip_rows = skip_row.size();
  ppi::ParseParams p;
  pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, n_cols, col_types, out_offsets, out_chars,
                                out_typed, records_capacity, chars_capacity, d_status, &p);
  if (rc != PP_OK) return rc;
  if (o.col_default)
    for (int c = 0; c < n_cols; ++c) p.defval[c] = o.col_default[c];
  Allocs A(stream);
  cudaError_t e;
  const uint8_t* in = d_in;
  uint64_t n = n_bytes;

  // ---- skipped rows: compact the input first
  if (o.n_skip_rows && n) {
    const int rd = rd_byte(dfa);
    if (rd < 0) return PP_EINVAL;
    const uint64_t nb = (n + RB - 1) / RB, nr = o.n_skip_rows;
    uint32_t* cnt;
    uint64_t *rows_before, *rows, *rstart, *rlen, *skipped;
    uint8_t* out;
    if ((e = A.get(reinterpret_cast<void**>(&cnt), nb * 4)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&rows_before), (nb + 1) * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&rows), nr * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&rstart), nr * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&rlen), nr * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&skipped), (nr + 1) * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&out), n)) != cudaSuccess)
      return rc_of(e);
    if ((e = cudaMemcpyAsync(rows, o.skip_rows, nr * 8, cudaMemcpyHostToDevice, stream)) !=
        cudaSuccess)
      return rc_of(e);
    row_count_kernel<<<unsigned(std::min<uint64_t>(nb, 4096)), 256, 0, stream>>>(in, n, uint8_t(rd),
                                                                                cnt, nb);
    exclusive_scan_kernel<<<1, SCAN_T, 0, stream>>>(nullptr, cnt, nb, rows_before);
    row_range_kernel<<<unsigned((nr + 255) / 256), 256, 0, stream>>>(in, n, uint8_t(rd),
                                                                     rows_before, nb, rows, nr,
                                                                     rstart, rlen);
    exclusive_scan_kernel<<<1, SCAN_T, 0, stream>>>(rlen, nullptr, nr, skipped);
    drop_ranges_kernel<<<unsigned(std::min<uint64_t>((n / 16 + 255) / 256 + 1, 65535)), 256, 0,
                         stream>>>(in, n, rstart, rlen, skipped, nr, out);
    if ((e = cudaGetLastError()) != cudaSuccess) return rc_of(e);
    uint64_t dropped = 0;  // the compacted size decides the tiling: wait for it
    if ((e = cudaMemcpyAsync(&dropped, skipped + nr, 8, cudaMemcpyDeviceToHost, stream)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
      return rc_of(e);
    in = out;
    n -= dropped;
    rc = ppi::parse_prepare(in, n, dfa, n_cols, col_types, out_offsets, out_chars, out_typed,
                            records_capacity, chars_capacity, d_status, &p);
    if (rc != PP_OK) return rc;
    if (o.col_default)
      for (int c = 0; c < n_cols; ++c) p.defval[c] = o.col_default[c];
  }

  // ---- records not emitted: the bitmap and its prefix sums
  const bool reject = (o.flags & PP_PARSE_REJECT) != 0;
  if (reject || o.n_skip_records) {
    const uint64_t n_bits = n + 2;  // records of the input (at most n + 1)
    const uint64_t n_groups = (n_bits + 255) / 256, n_words = n_groups * 8;
    uint32_t* bits;
    uint64_t *pre, *gcnt, *list = nullptr;
    if ((e = A.get(reinterpret_cast<void**>(&bits), n_words * 4)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&gcnt), n_groups * 8)) != cudaSuccess ||
        (e = A.get(reinterpret_cast<void**>(&pre), (n_groups + 1) * 8)) != cudaSuccess)
      return rc_of(e);
    if ((e = cudaMemsetAsync(bits, 0, n_words * 4, stream)) != cudaSuccess) return rc_of(e);
    if (o.n_skip_records) {
      if ((e = A.get(reinterpret_cast<void**>(&list), o.n_skip_records * 8)) != cudaSuccess ||
          (e = cudaMemcpyAsync(list, o.skip_records, o.n_skip_records * 8, cudaMemcpyHostToDevice,
                               stream)) != cudaSuccess)
        return rc_of(e);
      scatter_bits_kernel<<<unsigned((o.n_skip_records + 255) / 256), 256, 0, stream>>>(
          list, o.n_skip_records, n_bits, bits);
    }
    if (reject && n) {
      // status pass: the tile kernel without outputs marks the records whose
      // field count is not n_cols
      std::vector<pp_coltype> skip(size_t(n_cols), PP_COL_SKIP);
      ppi::ParseParams q;
      rc = ppi::parse_prepare(in, n, dfa, n_cols, skip.data(), nullptr, nullptr, nullptr, 0,
                              nullptr, d_status, &q);
      if (rc != PP_OK) return rc;
      q.mark_bits = bits;
      void* scr;
      if ((e = A.get(&scr, ppi::parse_scratch_bytes(q.n_tiles, 0))) != cudaSuccess) return rc_of(e);
      ppi::parse_scratch_carve(scr, q.n_tiles, 0, &q.s);
      if ((e = ppi::launch_parse(q, stream)) != cudaSuccess) return rc_of(e);
    }
    group_count_kernel<<<unsigned((n_groups + 255) / 256), 256, 0, stream>>>(bits, n_groups, gcnt);
    exclusive_scan_kernel<<<1, SCAN_T, 0, stream>>>(gcnt, nullptr, n_groups, pre);
    if ((e = cudaGetLastError()) != cudaSuccess) return rc_of(e);
    p.drop_bits = bits;
    p.drop_pre = pre;
    p.skip_list = list;
    p.n_skip = o.n_skip_records;
  }

  // ---- the parse
  const int ns = ppi::parse_ns_width(p.n_str);
  void* scratch;
  if ((e = A.get(&scratch, ppi::parse_scratch_bytes(p.n_tiles, ns, p.enc != 0))) != cudaSuccess)
    return rc_of(e);
  ppi::parse_scratch_carve(scratch, p.n_tiles, ns, &p.s, p.enc != 0);
  return rc_of(ppi::launch_parse(p, stream));
}

extern "C" pp_rc pp_infer_types(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                                int n_cols, int32_t* d_types, pp_status* d_status,
                                cudaStream_t stream) {
  if (!d_types || (dfa && dfa->encoding != PP_ENC_BYTES)) return PP_EINVAL;
  std::vector<pp_coltype> skip(size_t(n_cols > 0 ? n_cols : 1), PP_COL_SKIP);
  ppi::ParseParams p;
  const pp_rc rc = ppi::parse_prepare(d_in, n_bytes, dfa, n_cols, skip.data(), nullptr, nullptr,
                                      nullptr, 0, nullptr, d_status, &p);
  if (rc != PP_OK) return rc;
  // every column classified by the tile pass's number phase, nothing stored
  for (int c = 0; c < n_cols; ++c) p.coltype[c] = ppi::COL_INFER;
  p.has_out = 1;
  Allocs A(stream);
  cudaError_t e;
  uint32_t* codes;
  void* scratch;
  if ((e = A.get(reinterpret_cast<void**>(&codes), size_t(n_cols) * 4)) != cudaSuccess ||
      (e = A.get(&scratch, ppi::parse_scratch_bytes(p.n_tiles, 0))) != cudaSuccess)
    return rc_of(e);
  if ((e = cudaMemsetAsync(codes, 0, size_t(n_cols) * 4, stream)) != cudaSuccess) return rc_of(e);
  p.infer_out = codes;
  ppi::parse_scratch_carve(scratch, p.n_tiles, 0, &p.s);
  if ((e = ppi::launch_parse(p, stream)) != cudaSuccess) return rc_of(e);
  return rc_of(ppi::launch_infer_finish(codes, d_types, n_cols, stream));
}
