/*
 * pp.h — C ABI of libpp, a GB300 (sm_103a) library for massively parallel
 * parsing of delimiter-separated raw data with a DFA, after "ParPaRaw:
 * Massively Parallel Parsing of Delimiter-Separated Raw Data".
 *
 * What is computed (ParPaRaw, Section 3): every chunk of the input runs one
 * DFA instance per state, giving a state-transition vector (Section 3.1,
 * Figure 2); an exclusive scan with the composite operation gives each
 * chunk its true start state; a single DFA run then tags each byte as field
 * delimiter, record delimiter, control symbol or value (Section 3.1, the
 * three bitmap indexes); record counts and absolute/relative column offsets
 * are scanned (Section 3.2, Figure 4); values are emitted per column
 * (Section 3.3, Figure 5) — here directly as Arrow-style int32 offsets plus
 * chars for string columns (the Arrow layout as described in the libcudf
 * string-column article: offsets[0] = 0, offsets[i+1] - offsets[i] = size
 * of row i, last offset = chars size) and as dense arrays for numeric
 * columns (type conversion, Section 3.3; empty field = default value 0,
 * Section 4.3).
 *
 * Conventions for every entry point:
 *  - Per-device set-up (kernel attributes, SM counts) is done once per
 *    device ordinal, on the first call made with that device current, and
 *    is safe to reach from several host threads at once.  It applies to
 *    the device's primary context, the one the CUDA runtime API uses.
 *  - Pointers named d_* and out_* are DEVICE pointers; everything else
 *    (descriptors, column-type arrays, capacity arrays, pointer arrays) is
 *    HOST memory, read during the call only.
 *  - The caller owns all input and output buffers.  Scratch for the
 *    cross-block scan is allocated stream-ordered on `stream`
 *    (cudaMallocAsync) and released stream-ordered before return.
 *  - All device work is enqueued on `stream`; no call synchronises the
 *    host except where stated.
 *  - The return code covers argument checks and CUDA launch/allocation
 *    errors only.  Errors found in the data are reported in the device-side
 *    pp_status (error bitmask + the minimum byte offset of any data error).
 *  - Outputs are defined only when pp_status.error holds none of the fatal
 *    bits (PP_ERR_FATAL).  Every store is bounds-checked against the given
 *    capacities whatever the input.
 */
#ifndef PP_H
#define PP_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PP_MAX_COLS 64
#define PP_MAX_STATES 16
#define PP_MAX_GROUPS 16

/* host return codes */
typedef enum {
  PP_OK = 0, PP_EINVAL = 1, PP_ECUDA = 2, PP_ENOMEM = 3, PP_ETOOLARGE = 4,
  PP_ECHUNK = 5 /* pp_parse_host: a record longer than the streaming chunk */
} pp_rc;

/* column kinds for pp_parse */
typedef enum {
  PP_COL_STRING = 0, /* Arrow int32 offsets[R+1] + uint8 chars          */
  PP_COL_INT8 = 1,   /* int8[R],  grammar [+-]?[0-9]+                   */
  PP_COL_INT32 = 2,  /* int32[R]                                        */
  PP_COL_INT64 = 3,  /* int64[R]                                        */
  PP_COL_FLOAT64 = 4,/* double[R], decimal grammar, within 1 ulp of the
                        correctly rounded value                          */
  PP_COL_SKIP = 5,   /* parsed for structure, not emitted               */
  PP_COL_TIMESTAMP = 6 /* int64[R]: a temporal field (ParPaRaw Section 3.3,
                        "numerical or temporal types") as seconds since
                        1970-01-01 00:00:00, proleptic Gregorian calendar,
                        no time zone.  Grammar YYYY-MM-DD or
                        YYYY-MM-DD HH:MM:SS with month 01-12, day within
                        the month, hour 00-23, minute and second 00-59;
                        anything else is PP_ERR_NUM_SYNTAX with value 0  */
} pp_coltype;

/* per-byte tags (ParPaRaw Section 3.1: record delimiter, field delimiter,
 * control symbol vs. value; plus "invalid" for transitions into the error
 * state, Section 4.3 "Validating format", and "begin" for lexers)         */
typedef enum {
  PP_TAG_DATA = 0,    /* part of a value                                 */
  PP_TAG_FD = 1,      /* field delimiter                                 */
  PP_TAG_RD = 2,      /* record delimiter                                */
  PP_TAG_CTRL = 3,    /* control symbol (quote, escape) — not a value    */
  PP_TAG_INVALID = 4, /* transition into / inside the invalid state      */
  PP_TAG_BEGIN = 5    /* first byte of a token (pp_tokenize DFAs)        */
} pp_tag;

/* pp_status.error bits */
#define PP_ERR_INVALID_INPUT 1    /* a transition into the invalid state    */
#define PP_ERR_BAD_END_STATE 2    /* input ends in a non-accepting state    */
#define PP_ERR_COLCOUNT 4         /* a record with != n_cols fields         */
#define PP_ERR_NUM_SYNTAX 8       /* numeric field does not match grammar   */
#define PP_ERR_NUM_OVERFLOW 16    /* integer out of range for its column    */
#define PP_ERR_CAPACITY 32        /* an output capacity was too small       */
#define PP_ERR_LOOKBACK_TIMEOUT 64/* a cross-block wait gave up (bounded)   */
#define PP_ERR_FATAL (PP_ERR_INVALID_INPUT | PP_ERR_BAD_END_STATE | \
                      PP_ERR_CAPACITY | PP_ERR_LOOKBACK_TIMEOUT)

/* Symbol encodings of the input (ParPaRaw Section 3.4: with a
 * variable-length encoding a symbol spans several bytes and may cross chunk
 * boundaries).
 *   PP_ENC_BYTES    every byte is a symbol (the default).
 *   PP_ENC_UTF8     a symbol is a byte that is not 0b10xxxxxx together with
 *                   the 0b10xxxxxx bytes after it; it is well formed if it
 *                   has the length its first byte announces, is not an
 *                   overlong form and is at most 0x10FFFF.
 *   PP_ENC_UTF16LE  2-byte little-endian units from the input's first byte;
 *                   a high surrogate followed by a low surrogate is one
 *                   4-byte symbol; an odd last byte is a symbol of its own.
 * With an encoding the DFA takes one transition per symbol, at the symbol's
 * last byte, so every offset the library reports for a symbol (a record
 * delimiter, an invalid transition) is that of its last byte.  A value
 * keeps all bytes of its value symbols; the other bytes of a multi-byte
 * delimiter or control symbol are dropped like a control symbol.
 * Symbol groups: a code point below 0x80 takes byte_to_group[code point],
 * the code points listed in sym_cp take sym_group, and every other symbol
 * (ill-formed ones too) takes byte_to_group[0x80].                        */
#define PP_ENC_BYTES 0
#define PP_ENC_UTF8 1
#define PP_ENC_UTF16LE 2
#define PP_MAX_SYMS 8

/* Description of a DFA over bytes or symbols (ParPaRaw Section 5, Table 1:
 * symbols with identical transitions are collapsed into symbol groups, and
 * the transition table is stored with one row per symbol group).          */
typedef struct {
  uint8_t n_states;       /* |S|, 1..16                                    */
  uint8_t n_groups;       /* symbol groups, 1..16                          */
  uint8_t start_state;    /* state of the sequential DFA at byte 0         */
  uint8_t invalid_state;  /* absorbing error state, or 0xFF for none       */
  uint16_t accept_mask;   /* bit s set: s is an accepting end state        */
  uint8_t background_group; /* a group whose transition is idempotent and
                               whose bytes are never delimiters/controls, or
                               0xFF; lets the tagger skip runs of it        */
  uint8_t encoding;       /* PP_ENC_*: pp_parse, pp_parse_ex (without
                             skipped rows) and pp_parse_noalloc take every
                             encoding, with string, integer, float and skip
                             columns; the other entry points, and timestamp
                             columns, take PP_ENC_BYTES only (else
                             PP_EINVAL)                                    */
  uint8_t byte_to_group[256];
  uint8_t delta[PP_MAX_GROUPS][PP_MAX_STATES]; /* delta[group][state]       */
  uint8_t tag[PP_MAX_STATES][PP_MAX_GROUPS];   /* tag[state_before][group]  */
  /* pp_tokenize only: token id from the state after the token's last byte;
   * 0xFE means "take byte_token_id[first byte of the token]"             */
  uint8_t token_id[PP_MAX_STATES];
  uint8_t byte_token_id[256];
  /* encodings other than PP_ENC_BYTES: code points of at least 0x80 with a
   * group of their own (distinct, at most 0x10FFFF, no surrogates)        */
  uint8_t n_syms;
  uint8_t sym_group[PP_MAX_SYMS];
  uint8_t reserved2[3];
  uint32_t sym_cp[PP_MAX_SYMS];
} pp_dfa_desc;

/* Device-resident result status.  The caller allocates it; every call
 * initialises it on `stream` before any other device work.               */
typedef struct {
  int32_t error;                 /* 0 or PP_ERR_* bitmask                  */
  int32_t reserved;
  uint64_t first_error_offset;   /* min byte offset over all data errors
                                    (INVALID_INPUT at the offending byte,
                                    BAD_END_STATE at n_bytes, COLCOUNT at
                                    the record's terminator, NUM_* at the
                                    field's first byte); UINT64_MAX if none */
  uint64_t n_records;            /* pp_parse                               */
  uint64_t n_tokens;             /* pp_tokenize                            */
  uint64_t chars_len[PP_MAX_COLS]; /* pp_parse: chars of column c (string
                                    columns; 0 for the others)             */
  uint64_t n_dropped;            /* pp_parse_ex: records of the input not
                                    emitted (skipped or rejected)          */
} pp_status;

/*
 * pp_parse — parse delimiter-separated input into columns.
 *   d_in            device, n_bytes bytes of raw input (any alignment).
 *   dfa             host; a DFA with at most 4 live states plus (optionally)
 *                   one absorbing invalid state with index 4, tags FD/RD/
 *                   CTRL/DATA/INVALID (e.g. built by pp_desc_csv).
 *   n_cols          1..PP_MAX_COLS; col_types[n_cols] host.
 *   out_offsets[c]  device int32[records_capacity+1] for PP_COL_STRING
 *                   columns, else ignored (may be NULL).
 *   out_chars[c]    device uint8[chars_capacity[c]] for string columns.
 *   out_typed[c]    device array of records_capacity elements of the
 *                   column's type for numeric and timestamp columns (int64
 *                   for PP_COL_TIMESTAMP).
 *   chars_capacity  host array of n_cols sizes (string columns only).
 *   d_status        device pp_status.
 * Passing NULL for every out_offsets/out_chars/out_typed pointer is allowed
 * (a sizing pass): nothing is written except d_status, whose n_records and
 * chars_len then give exact sizes.
 * Semantics (ParPaRaw Sections 3-4): a record ends at every record
 * delimiter; a non-empty tail without one is one more record; an empty line
 * is a record with one empty field; records with != n_cols fields set
 * PP_ERR_COLCOUNT, extra fields are dropped and missing ones take the
 * default (empty string / 0).  String values are the value bytes only
 * (enclosing quotes dropped, a doubled quote yields one quote).
 * Inputs of 2^40 bytes (1 TiB) or more return PP_ETOOLARGE.
 * Returns PP_EINVAL for bad arguments, PP_ENOMEM / PP_ECUDA on CUDA errors.
 */
pp_rc pp_parse(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
               const pp_coltype* col_types, int32_t* const out_offsets[],
               uint8_t* const out_chars[], void* const out_typed[],
               size_t records_capacity, const size_t chars_capacity[],
               pp_status* d_status, cudaStream_t stream);

/* pp_parse_ex options (ParPaRaw Section 4).  A zero-initialised struct (or
 * a NULL pointer) gives pp_parse's behaviour. */
#define PP_PARSE_REJECT 1u  /* records whose field count is not n_cols are not
                               emitted (they still set PP_ERR_COLCOUNT)     */
typedef struct {
  uint32_t flags;               /* PP_PARSE_* bits                            */
  uint32_t reserved;            /* 0                                          */
  const uint64_t* col_default;  /* host, n_cols entries, or NULL: the bits
                                   stored for an empty or missing field of a
                                   numeric or timestamp column (int64 two's
                                   complement, binary64 bits or seconds;
                                   truncated to int8/int32 columns) instead of
                                   0.  Section 4, "Default values for empty
                                   strings".  String columns keep the empty
                                   string.                                    */
  const uint64_t* skip_records; /* host, ascending indices of records not to
                                   emit (counted in the input after skipped
                                   rows), or NULL.  Section 4, "Skipping
                                   records and selecting columns": their
                                   fields are irrelevant (not converted, no
                                   column-count check).                       */
  uint64_t n_skip_records;
  const uint64_t* skip_rows;    /* host, ascending indices of rows (lines:
                                   bytes up to and including each record-
                                   delimiter byte, whatever the quoting, plus
                                   a last line without one) removed before
                                   parsing, or NULL.  Section 4, "Skipping
                                   rows".  Error offsets then refer to the
                                   input without those rows.                  */
  uint64_t n_skip_rows;
} pp_parse_opts;

/*
 * pp_parse_ex — pp_parse with the options above.  Emitted records are
 * numbered 0.. in input order without the dropped ones; n_records counts
 * the emitted records and n_dropped the others.
 *   Extra device memory (stream-ordered): with skip_rows, a copy of the
 *   input without those rows (n_bytes); with PP_PARSE_REJECT or
 *   skip_records, a dropped-record bitmap and its prefix sums (about
 *   n_bytes / 6) and one more pass over the input for PP_PARSE_REJECT.
 *   skip_rows needs the record delimiter to be the byte the descriptor's
 *   PP_TAG_RD transitions read (as for pp_desc_csv / pp_desc_csv_crlf).
 * Returns as pp_parse; PP_EINVAL also for unsorted skip lists.
 */
pp_rc pp_parse_ex(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                  const pp_coltype* col_types, const pp_parse_opts* opts,
                  int32_t* const out_offsets[], uint8_t* const out_chars[],
                  void* const out_typed[], size_t records_capacity,
                  const size_t chars_capacity[], pp_status* d_status, cudaStream_t stream);

/*
 * pp_parse_host — pp_parse of an input in HOST memory into outputs in HOST
 * memory, streamed through the device in chunks (the streaming set-up of
 * ParPaRaw Section 4: partitions move to the device while earlier ones are
 * parsed and their results move back).
 *   h_in, h_offsets[], h_chars[], h_typed[], h_status: host memory, laid
 *   out and filled exactly as pp_parse fills its device buffers (offsets
 *   [records + 1] int32 per string column, chars, one typed array per
 *   numeric column, and the status).  Page-locked (pinned) host memory lets
 *   the copies run asynchronously and overlap the parse; pageable memory
 *   works, with the copies staged by the CUDA driver.
 *   records_capacity, chars_capacity[]: as in pp_parse, for the whole input.
 *   chunk_bytes: bytes of new input per chunk (rounded up to a multiple of
 *   pp_tile_bytes(); 0 = 128 MiB).  Each chunk after the first begins with
 *   the bytes of the record left unfinished at the end of the one before,
 *   so a record may be at most chunk_bytes long; a longer one stops the
 *   call with PP_ECHUNK (h_status then holds the records emitted so far
 *   and PP_ERR_CAPACITY at the offending record).
 *   stream: parses run on it; the copies in each direction run on a
 *   stream of their own that the call creates.  The call returns once
 *   every result is in host memory.
 *   Device memory: two input buffers of 2 x chunk_bytes, two staging
 *   buffers of chunk_bytes and two sets of output buffers, each for
 *   min(records_capacity, 2 x chunk_bytes) + 1 records (chars per string
 *   column min(chars_capacity, 2 x chunk_bytes)), from the stream-ordered
 *   allocator.  The call sets the device's default memory pool to keep
 *   freed memory (release threshold: unlimited), so later calls reuse it.
 * Returns PP_EINVAL for bad arguments, PP_ECHUNK as above, PP_ENOMEM /
 * PP_ECUDA on CUDA errors.
 */
pp_rc pp_parse_host(const uint8_t* h_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                    const pp_coltype* col_types, int32_t* const h_offsets[],
                    uint8_t* const h_chars[], void* const h_typed[], size_t records_capacity,
                    const size_t chars_capacity[], pp_status* h_status, size_t chunk_bytes,
                    cudaStream_t stream);

/*
 * pp_tokenize_host — pp_tokenize of an input in HOST memory into triples in
 * HOST memory, streamed through the device in chunks as pp_parse_host does.
 *   h_in, h_token_id, h_start, h_len, h_status: host memory (pinned for
 *   overlapped copies), filled as pp_tokenize fills its device buffers;
 *   tokens_capacity = 0 with null outputs counts the tokens only.
 *   chunk_bytes: as for pp_parse_host.  Each chunk after the first begins
 *   at the start of the token left open at the end of the one before, in
 *   the DFA state that token started from, so a token may be at most
 *   chunk_bytes long; a longer one returns PP_ECHUNK.
 *   Device memory: the input buffers of pp_parse_host, plus two sets of
 *   triples for min(tokens_capacity, 2 x chunk_bytes) + 1 tokens.
 * Returns PP_EINVAL for bad arguments, PP_ECHUNK as above, PP_ENOMEM /
 * PP_ECUDA on CUDA errors.
 */
pp_rc pp_tokenize_host(const uint8_t* h_in, size_t n_bytes, const pp_dfa_desc* dfa,
                       uint8_t* h_token_id, uint64_t* h_start, uint32_t* h_len,
                       size_t tokens_capacity, pp_status* h_status, size_t chunk_bytes,
                       cudaStream_t stream);

/* Size of pp_parse_noalloc's fixed scratch buffer (per device). */
#define PP_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * pp_parse_noalloc — pp_parse without allocation: its cross-tile scratch
 * (tile vectors and states, look-back flags and aggregates) lives in a buffer of
 * PP_NOALLOC_SCRATCH_BYTES compiled into the library, one per device.  The
 * ParPaRaw paper has no counterpart; this is an integration entry point
 * for callers that cannot allocate device memory per call (devices or
 * driver set-ups without stream-ordered memory pools, where pp_parse's
 * cudaMallocAsync fails; services whose device memory is fixed at
 * start-up).
 *   Arguments, semantics, outputs and d_status: exactly those of pp_parse.
 *   Limit: the scratch needed is about 22 bytes per 16 KiB tile of input
 *   without string columns and 4 + 16 x w bytes more with them, w being the
 *   string-column count rounded up to 4, 8 or 16, plus up to 128 KiB for
 *   the queue of long numeric fields; 4 MiB therefore holds inputs up to
 *   about 2.9 GiB without string columns, 710 MiB with 1 to 4, 410 MiB with
 *   5 to 8 and 225 MiB with 9 to 16 string columns.  A larger input returns
 *   PP_ETOOLARGE before any CUDA call.
 *   First call on each device: it looks up the buffer's address
 *   (cudaGetSymbolAddress; this can load the library's device code) and
 *   sets kernel attributes.  Make that first call before any stream
 *   capture starts on the device.  The address is kept per device ordinal
 *   and belongs to the device's primary context, the one the CUDA runtime
 *   API uses; a caller that switches the device to another context (driver
 *   API) must not call this entry point from that context.
 *   Calls share the buffer: two calls in flight on one device at the same
 *   time (on different streams, or from host threads with no ordering
 *   between them) race on it and corrupt each other's results.  Issue the
 *   calls on one stream, or order them by events or synchronisation.
 * Returns PP_EINVAL for bad arguments, PP_ETOOLARGE as above, PP_ENOMEM
 * when a launch reports cudaErrorMemoryAllocation (the kernels' own
 * resources; the call allocates no memory), PP_ECUDA on other CUDA errors.
 */
pp_rc pp_parse_noalloc(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                       const pp_coltype* col_types, int32_t* const out_offsets[],
                       uint8_t* const out_chars[], void* const out_typed[],
                       size_t records_capacity, const size_t chars_capacity[],
                       pp_status* d_status, cudaStream_t stream);

/*
 * pp_tokenize — run a general DFA (|S| <= 16) over the input and emit one
 * (token_id, start, len) triple per token, as struct-of-arrays.  A token
 * starts at byte 0 and at every byte whose tag is PP_TAG_BEGIN; its length
 * runs to the next token start (or n_bytes); its id is token_id[state after
 * its last byte] (the prefix-scan lexer of "Lexing on the GPU: the scan is
 * the easy part", section "A lexer is a prefix scan").
 *   out_token_id   device uint8[tokens_capacity]
 *   out_start      device uint64[tokens_capacity]
 *   out_len        device uint32[tokens_capacity]
 * NULL outputs with tokens_capacity 0 make a counting pass (n_tokens only).
 * Tokens beyond tokens_capacity are counted, not written (PP_ERR_CAPACITY).
 */
pp_rc pp_tokenize(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                  uint8_t* out_token_id, uint64_t* out_start, uint32_t* out_len,
                  size_t tokens_capacity, pp_status* d_status, cudaStream_t stream);

/*
 * pp_tags — test hook: per byte, the state of the sequential DFA before the
 * byte and the byte's tag (tag[state_before][group]), computed by the same
 * multi-instance DFA + composite scan as the parsers (ParPaRaw Section
 * 3.1).  d_state_before and d_tag are device uint8[n_bytes].  d_status gets
 * error/first_error_offset for INVALID_INPUT and BAD_END_STATE.
 */
pp_rc pp_tags(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
              uint8_t* d_state_before, uint8_t* d_tag, pp_status* d_status,
              cudaStream_t stream);

/*
 * pp_count_byte — *d_count = number of bytes equal to `value` in d_in
 * (uint64, device).  With value = the record delimiter, *d_count + 1 bounds
 * the record count of any input, which is how callers size pp_parse
 * outputs without a sizing pass.
 */
pp_rc pp_count_byte(const uint8_t* d_in, size_t n_bytes, uint8_t value, uint64_t* d_count,
                    cudaStream_t stream);

/*
 * pp_count_fields — column-count inference (ParPaRaw Section 4, "Inferring
 * or validating number of columns"): the fewest and the most fields of any
 * record of the input, for a caller without a schema or one that wants to
 * validate it before pp_parse.  A record has one more field than field
 * delimiters; a non-empty tail without a record delimiter is one more
 * record (as in pp_parse).  Each tile reduces its chunks' (delimiters
 * before the first record delimiter, after the last, fewest and most fields
 * in between) in order, and one block combines the tiles.
 *   d_in      device, n_bytes bytes (any alignment).
 *   dfa       host; the same descriptors as pp_parse takes.
 *   d_fields  device uint64[2]: [0] fewest, [1] most fields per record
 *             (both 0 for an input without records).
 *   d_status  device; error bits as pp_parse (invalid input, a
 *             non-accepting end state; with a fatal bit d_fields is
 *             unspecified) and n_records.
 * Scratch about 25 bytes per 16 KiB tile, taken stream-ordered
 * (cudaMallocAsync) and freed the same way; asynchronous on `stream`.
 * Inputs up to 64 GiB (2^36 bytes); larger ones return PP_ETOOLARGE.
 * Returns PP_EINVAL for bad arguments, PP_ENOMEM / PP_ECUDA on CUDA errors.
 */
pp_rc pp_count_fields(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                      uint64_t* d_fields, pp_status* d_status, cudaStream_t stream);

/*
 * pp_infer_types — numeric type inference (ParPaRaw Section 4, "Type
 * inference"): for each of the first n_cols columns, the smallest of
 * PP_COL_INT8 < PP_COL_INT32 < PP_COL_INT64 < PP_COL_FLOAT64 <
 * PP_COL_STRING that backs every field of the column.  A field's value
 * bytes (quotes dropped, as pp_parse reads them) take int8/int32/int64 when
 * they match [+-]?[0-9]+ within that range, float64 when they match the
 * float grammar of PP_COL_FLOAT64 or are an integer beyond int64, and
 * string otherwise; empty and missing fields constrain nothing, so a
 * column without a non-empty field is PP_COL_INT8.  Fields past n_cols
 * are ignored.  Each tile classifies its fields and reduces them per
 * column; the tiles combine by an atomic maximum.
 *   d_in      device, n_bytes bytes (any alignment); dfa as for pp_parse.
 *   n_cols    1..PP_MAX_COLS (for instance the most fields per record from
 *             pp_count_fields).
 *   d_types   device int32[n_cols]: pp_coltype values.
 *   d_status  device; PP_ERR_INVALID_INPUT and PP_ERR_BAD_END_STATE as
 *             pp_parse (records need not have n_cols fields: no
 *             PP_ERR_COLCOUNT; no PP_ERR_NUM_*), and n_records.
 * Scratch as pp_parse, stream-ordered; asynchronous on `stream`.
 * Returns PP_EINVAL for bad arguments, PP_ENOMEM / PP_ECUDA on CUDA errors.
 */
pp_rc pp_infer_types(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa, int n_cols,
                     int32_t* d_types, pp_status* d_status, cudaStream_t stream);

/*
 * pp_desc_csv — build the quoted-CSV DFA (RFC-4180 style quoting) with
 * states EOR=0 (at a field/record boundary, the start state), FLD=1 (inside
 * an unquoted field), ENC=2 (inside quotes), ESC=3 (a quote seen inside
 * quotes), INV=4 (invalid, absorbing; ParPaRaw Section 3.1 names reading a
 * quote in FLD as invalid).  fd, rd and quote must be distinct.
 * Accepting end states: EOR, FLD, ESC.  Host only.
 */
pp_rc pp_desc_csv(pp_dfa_desc* out, uint8_t fd, uint8_t rd, uint8_t quote);

/*
 * pp_desc_csv_enc — the same quoted-CSV DFA over the symbols of a
 * variable-length encoding (encoding PP_ENC_UTF8 or PP_ENC_UTF16LE; ParPaRaw
 * Section 3.4): fd, rd and quote are code points (distinct, at most
 * 0x10FFFF, no surrogates), any of them may take several bytes.  Host only.
 */
pp_rc pp_desc_csv_enc(pp_dfa_desc* out, int encoding, uint32_t fd, uint32_t rd, uint32_t quote);

/*
 * pp_desc_csv_crlf — the same DFA for CRLF line ends: the record delimiter
 * is LF (0x0A), and a carriage return (0x0D) outside quotes is a control
 * symbol, dropped from the value, after which the field stays open (EOR,
 * FLD and ESC go to FLD on CR; inside quotes a CR is data).  The pages name
 * no line-end convention; ParPaRaw Section 4 ("Validating format") notes
 * that simulating the DFA allows such parsing rules.  fd and quote must be
 * distinct and neither may be LF or CR.  Host only; PP_EINVAL otherwise.
 */
pp_rc pp_desc_csv_crlf(pp_dfa_desc* out, uint8_t fd, uint8_t quote);

/*
 * pp_desc_json_lexer — build the 16-state JSON-like lexer DFA used by
 * pp_tokenize (whitespace runs, punctuation {}[],:, strings with backslash
 * escapes, integers, fractions and exponents).  Token ids: '{'0 '}'1 '['2
 * ']'3 ','4 ':'5 string 6 integer 7 float 8 whitespace 9, 255 invalid.
 * Host only.  Source: "Lexing on the GPU: the scan is the easy part",
 * section "A lexer is a prefix scan" (a lexer as one DFA whose transitions
 * mark token starts); the state table is this library's own, since the page
 * gives the scheme and not a table.
 */
pp_rc pp_desc_json_lexer(pp_dfa_desc* out);

/* Human-readable text for a pp_rc value. */
const char* pp_strerror(int code);

/* Tile size in bytes used by the cross-block scan (for tests that place
 * adversarial inputs at tile boundaries). */
size_t pp_tile_bytes(void);

/* Test/debug hook: number of polls a cross-block wait makes before it gives
 * up and reports PP_ERR_LOOKBACK_TIMEOUT (0 restores the default, about one
 * second of polling).  Process-wide; affects calls made afterwards. */
void pp_debug_set_spin_limit(uint32_t polls);

/* Test hook for the bounded waits: while on, the first tile of pp_parse's
 * tile pass posts nothing to its cross-tile look-backs, so the waits of the
 * tiles after it run out after the spin limit and the call reports
 * PP_ERR_LOOKBACK_TIMEOUT (fatal: outputs unspecified).  No wait is left
 * unbounded; the device stays usable.  Process-wide. */
void pp_debug_set_withhold(int on);

/* Benchmark hook: with n_calls > 0, the next n_calls pp_parse or
 * pp_tokenize calls record CUDA events on their stream around each of their
 * kernels.  0 stops recording and frees the events.
 * Process-wide; not thread-safe.  Returns PP_ECUDA if events cannot be
 * created. */
pp_rc pp_debug_stage_timing(int n_calls);

/* Kernel durations of the recorded calls: out[PP_STAGES*i + k] =
 * milliseconds of kernel k of call i.  pp_parse: 0 init, 1 tile transition
 * vectors, 2 tile start states, 3 tile pass (tagging, indices, columns and
 * conversion), 4 long numeric fields (a warp per queued field).
 * pp_tokenize: 0 init, 1 transition vectors, 2 state scan, 3 count pass,
 * 4 count scan, 5 emit pass.  Entries a call does not use are 0.  Waits for
 * the events.  Returns the number of calls written (at most max_calls), or
 * -1 on a CUDA error. */
#define PP_STAGES 6
int pp_debug_stage_ms(float* out, int max_calls);

/* Test hook: the tag bitmaps the tile pass of pp_parse computes (ParPaRaw
 * Section 3.1, the bitmap indexes): for the 32-byte chunk k of the input,
 * d_bits[3k] has bit j set if byte 32k + j is a field delimiter, d_bits[3k+1]
 * a record delimiter, d_bits[3k+2] a control symbol.  d_bits: device,
 * 3 * ceil(n_bytes / 32) words, written for every chunk.  Runs the parse's
 * kernels with no outputs; data errors go to d_status as for pp_parse.
 * Returns PP_EINVAL on a bad argument, PP_ENOMEM / PP_ECUDA on CUDA errors. */
pp_rc pp_debug_parse_tags(const uint8_t* d_in, size_t n_bytes, const pp_dfa_desc* dfa,
                          uint32_t* d_bits, pp_status* d_status, cudaStream_t stream);

/* Test hook: *out (if not NULL) = the number of numeric fields converted by
 * the long-field pass (a warp per field longer than 256 bytes) on the
 * current device since the last reset; reset != 0 then sets it to 0.
 * Synchronous (waits for the device).  Returns PP_ECUDA on a CUDA error. */
pp_rc pp_debug_long_fields(uint64_t* out, int reset);

#ifdef __cplusplus
}
#endif
#endif /* PP_H */
