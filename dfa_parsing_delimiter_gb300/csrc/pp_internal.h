// Host/device shared definitions of libpp (not part of the public ABI).
#pragma once
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime_api.h>
#include "pp.h"

namespace ppi {

// ------------------------------------------------------- per-device set-up
// Kernel attributes (cudaFuncSetAttribute) and occupancy belong to a device
// (its primary context, the one the runtime API uses), so every launcher
// keeps its set-up per device ordinal.  DeviceOnce runs a set-up function
// once per device, safely for concurrent host threads: the state it fills
// is published by a release store and read after an acquire load.  A
// set-up that fails is tried again by the next call.
constexpr int MAX_DEVICES = 64;

// The current device's ordinal (cudaErrorInvalidDevice beyond MAX_DEVICES).
cudaError_t current_device(int* dev);
// Streaming multiprocessors of the current device.
cudaError_t sm_count(int* out);

class DeviceOnce {
 public:
  template <class F>
  cudaError_t run(int dev, F&& setup) {
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> g(m_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = setup(dev);
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  std::mutex m_;
  std::atomic<bool> done_[MAX_DEVICES] = {};
};

constexpr int MAX_STR_COLS = 16;  // string columns per pp_parse call
constexpr uint8_t COL_INFER = 7;  // internal column kind: type inference only

// Scratch of one pp_parse call (device memory).
//   tile_stv, tile_state: per tile, its transition vector and its true start
//         state (from the tile-state scan, whose look-back words are
//         tstate_words).
//   v2_desc: the tile pass's look-back over (record count, last
//         terminator, column offset): a 16-byte descriptor per tile.
//   c_*:  its look-back over the value bytes per string column: per tile a
//         flag and ns-word aggregate / inclusive prefix (null without string
//         columns).
// A numeric field queued for conversion by a warp (long fields): output row,
// input byte range, column | type << 8, and the DFA state at its start
// (LONG_STATE | state) when known, else 0 (found from its tile's start).
struct LongField { uint64_t rec, start, end; uint32_t col, state; };
constexpr uint32_t LONG_STATE = 0x80000000u;
constexpr uint32_t LONG_CAP = 4096;  // queued fields per call, at most
constexpr uint32_t SYM_LAST = 128, SYM_MID = 144;  // symbol codes (see ParseParams::enc)

struct ParseScratch {
  uint32_t* counters;       // [0] tile tickets, [2] column-count end flag, [3] tile-state scan
                            // tickets, [4] queued long fields, [5] queued fields begun in an
                            // earlier tile (encodings; at long_q[long_cap ...])
  LongField* long_q;        // [long_cap] (null: no queue, every field converted by its lane)
  uint32_t long_cap;
  uint32_t* tile_stv;       // [n_tiles]
  uint8_t* tile_state;      // [n_tiles]
  unsigned long long* tstate_words;  // [n_tstate_blocks]
  uint32_t n_tstate_blocks;
  uint64_t* v2_desc;        // [n_tiles][2]
  uint32_t* c_flag;         // [n_tiles]
  uint64_t* c_agg;          // [n_tiles][ns]
  uint64_t* c_inc;
};

struct ParseParams {
  const uint8_t* in;
  uint64_t n;
  uint32_t n_tiles;
  uint32_t spin_limit;
  uint32_t dbg_withhold;  // test hook: the first tile posts nothing to the look-backs
  uint32_t* dbg_tags;     // test hook, or null: per 32-byte chunk the tile pass's
                          // field-delimiter, record-delimiter and control bitmaps
  uint32_t lut[256];      // per byte (or symbol code): STV selector, next-state/tag fields, special bit
  // Inputs in an encoding (PP_ENC_UTF8, PP_ENC_UTF16LE): lut is indexed by
  // symbol code (a one-byte symbol below 0x80: the byte; SYM_LAST + group:
  // the last byte of a longer symbol; SYM_MID + group: its other bytes).
  uint8_t enc;            // PP_ENC_*
  uint8_t sym_n;          // code points with a group of their own
  uint8_t sym_dflt;       // group of every other symbol of 0x80 and above
  uint8_t sym_b2g[0x80];  // group of the code points below 0x80
  uint8_t sym_g[PP_MAX_SYMS];
  uint32_t sym_cp[PP_MAX_SYMS];
  uint32_t bg_next;       // nibble s = delta[background][s], s = 0..4
  uint32_t sticky;        // state whose non-inert groups set LUT bit 30 (4: none)
  uint16_t accept_mask;
  uint8_t start_state;
  uint8_t has_inv;        // state 4 is the absorbing invalid state
  int32_t n_cols;
  int32_t n_str;
  int32_t has_out;
  uint64_t strmask;             // bit c: column c is a string column
  int8_t stridx[PP_MAX_COLS];   // column -> string index, or -1
  uint8_t strcol[MAX_STR_COLS]; // string index -> column
  uint8_t coltype[PP_MAX_COLS];
  int32_t* offsets[MAX_STR_COLS];
  uint8_t* chars[MAX_STR_COLS];
  uint64_t chars_cap[MAX_STR_COLS];
  void* typed[PP_MAX_COLS];
  uint64_t rec_cap;
  pp_status* st;
  uint64_t defval[PP_MAX_COLS];  // bits stored for an empty or missing numeric field
  // pp_parse_ex with dropped records (skipped or rejected), else null:
  // bit r of drop_bits = record r of the input is not emitted; drop_pre[g]
  // = dropped records before group g (256 records, 8 words); skip_list[0,
  // n_skip) = the caller's sorted skipped records (no column-count check).
  const uint32_t* drop_bits;
  const uint64_t* drop_pre;
  const uint64_t* skip_list;
  uint64_t n_skip;
  // Status pass of PP_PARSE_REJECT (no outputs), else null: bit r is set
  // for every record r whose field count is not n_cols.
  uint32_t* mark_bits;
  // Type inference (pp_infer_types), else null: per column the largest
  // type code of its fields (columns of kind COL_INFER).
  uint32_t* infer_out;
  // Partial mode (streaming chunks), when not null: the input ends inside
  // an unfinished record, which is neither closed nor checked for an
  // accepting end state; st->n_records counts the complete records only,
  // and *record_end receives 1 + the position of the last record delimiter
  // (atomic maximum; the caller zeroes it).
  unsigned long long* record_end;
  ParseScratch s;
};

// bytes of scratch for n_tiles tiles and ns string columns (ns rounded to the
// kernel's instantiation width)
// sym: an input in an encoding (room in the long-field queue for one field
// per tile begun in an earlier tile)
size_t parse_scratch_bytes(uint32_t n_tiles, int ns, bool sym = false);
void parse_scratch_carve(void* base, uint32_t n_tiles, int ns, ParseScratch* out, bool sym = false);
int parse_ns_width(int n_str);

// init (counters, look-back flags, status), tile vectors, tile states, tile pass
cudaError_t launch_parse(const ParseParams& p, cudaStream_t stream);
// Stage timing (benchmark hook): stage_begin() opens the record of one
// call (false if recording is off or full); stage_mark(k) records its
// event k (0: before the first kernel, k: after the k-th).
bool stage_begin();
void stage_mark(int k, cudaStream_t stream);
// pp_parse's argument checks and kernel parameters (all but the scratch)
pp_rc parse_prepare(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                    const pp_coltype* col_types, int32_t* const out_offsets[],
                    uint8_t* const out_chars[], void* const out_typed[],
                    size_t records_capacity, const size_t chars_capacity[],
                    pp_status* d_status, ParseParams* out);
size_t parse_tile_bytes();
// column-count inference (pp_count_fields): scratch bytes for n_tiles tiles,
// and the launch (p from parse_prepare; its scratch is carved here)
size_t fields_scratch_bytes(uint32_t n_tiles);
cudaError_t launch_count_fields(ParseParams p, void* scratch, uint64_t* out, cudaStream_t stream);
// codes (0 empty .. 5 string) -> pp_coltype, n entries (type inference)
cudaError_t launch_infer_finish(const uint32_t* codes, int32_t* types, int n, cudaStream_t stream);

// ---------------------------------------------------------- pp_tags / tokenize
struct GenericDfa {
  uint8_t n_states;
  uint8_t start_state;
  uint8_t invalid_state;
  uint8_t pad;
  uint16_t accept_mask;
  uint8_t byte_to_group[256];
  uint8_t delta[PP_MAX_GROUPS][PP_MAX_STATES];
  uint8_t tag[PP_MAX_STATES][PP_MAX_GROUPS];
  uint8_t token_id[PP_MAX_STATES];
  uint8_t byte_token_id[256];
};

cudaError_t launch_tags(const uint8_t* in, uint64_t n, const GenericDfa& dfa,
                        uint8_t* state_before, uint8_t* tag, pp_status* st, void* scratch,
                        size_t scratch_bytes, cudaStream_t stream);
size_t tags_scratch_bytes(uint64_t n);

// carry_out: partial mode (see TokParams in pp_tokenize.cu), or null
cudaError_t launch_tokenize(const uint8_t* in, uint64_t n, const GenericDfa& dfa,
                            uint8_t* out_id, uint64_t* out_start, uint32_t* out_len,
                            uint64_t cap, pp_status* st, void* scratch, size_t scratch_bytes,
                            cudaStream_t stream, unsigned long long* carry_out = nullptr);
// pp_tokenize's checks of a descriptor, and its conversion
bool generic_dfa_ok(const pp_dfa_desc* d);
GenericDfa to_generic_dfa(const pp_dfa_desc* d);
size_t tokenize_scratch_bytes(uint64_t n);

cudaError_t launch_count_byte(const uint8_t* in, uint64_t n, uint8_t value, uint64_t* d_count,
                              cudaStream_t stream);

}  // namespace ppi
