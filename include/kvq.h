/*
 * kvq.h - C ABI of libkvq: a quantized KV cache for decode attention on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow five web pages on KV-cache quantization:
 *  - troisinh.com "KV Cache Quantization - Nen cache INT4/INT3" (sections
 *    "Tai sao Key va Value lai khac nhau?", "Mixed Precision", "Tai sao no
 *    hoat dong": per-channel keys, per-token values, Hadamard rotation,
 *    pre-RoPE keys rotated on the fly, hot 4-bit / cold 2-bit tokens);
 *  - nalar.dev "Kuantisasi KV Cache dengan Error Budget yang Eksplisit"
 *    (sections "Ukuran cache...", "Error pada key...", "Error pada value...",
 *    "Granularitas...", "Evaluasi...": the size law 2*L*T*H_kv*D, the scores
 *    s_i = q.k_i/sqrt(D), the output sum_i p_i v_i, a recent window kept at
 *    higher precision);
 *  - trefon.com "Matematyka cache KV" (sections "Bajty na token", the format
 *    table of "Przyklad: model 27B przy 262K", "Jak 4-bitowemu cache to
 *    uchodzi: najpierw obrot": block layouts Q8_0 34 B/32, Q4_0 18 B/32,
 *    66 B/128, 50 B/128; the randomized Walsh-Hadamard transform; attention
 *    in the rotated domain);
 *  - lehuy.net "NexusQuant" (section "Cac mo hinh duoc ho tro": split-half
 *    RoPE).
 *
 * Conventions shared by every entry point:
 *  - Ownership: the library never allocates device memory.  The caller owns
 *    every buffer and passes raw device pointers and a cudaStream_t (as
 *    void*; NULL means the legacy default stream).
 *  - Asynchrony: every call only enqueues work on the given stream, except
 *    kvq_read_device_status, which synchronizes that stream.
 *  - Errors: a kvq_status return.  Bad arguments are rejected on the host
 *    before anything is launched, with a message in kvq_last_error().  Bad
 *    runtime data found by a kernel (a length beyond capacity, a page id out
 *    of range) sets a bit of the device status word in the workspace and
 *    skips that piece of work; nothing traps.  The only waits are bounded
 *    waits of a kernel for its own copies into shared memory
 *    (KVQ_DEV_STALL when one runs out).
 *  - Head mapping: query head h reads kv head h / (H_q / H_kv).
 *  - Softmax scale: fixed at 1/sqrt(D).
 *
 * Cache representation (per sequence of T tokens, per layer and kv head):
 *  - tokens [q_end, T) stay unquantized in a 16-bit window (raw bits of the
 *    input dtype), q_end = max(0, floor((T - R)/Gamma)) * Gamma, where R is
 *    residual_window and Gamma is the token group of a per-channel format (1
 *    when both formats are per-token);
 *  - with hot_window W > 0: tokens [c_end, q_end) are in the hot formats
 *    (k_fmt, v_fmt) and [0, c_end) in the cold formats (k_cold, v_cold),
 *    c_end = max(0, floor((q_end - W)/Gamma)) * Gamma; a group that leaves
 *    the hot tier is requantized from its dequantized hot values;
 *  - with W = 0: tokens [0, q_end) are in k_fmt / v_fmt.
 *
 * Block: fp16 scale (little endian) then G*b/8 bytes of codes.  Absmax
 * scaling in fp32: amax = max|x|, scale = fp16_rn(min(amax/qmax, 65504)),
 * code = clamp(rint(x / float(scale)), -qmax, qmax), qmax = 2^(b-1) - 1,
 * all codes 0 when the scale is 0.  Packing: 8-bit two's complement;
 * 4-bit code+8, element 2i in the low nibble of byte i; 3-bit code+4,
 * eight values per 24-bit little-endian word, value j at bits [3j, 3j+3);
 * 2-bit code+2, value j of a byte at bits [2j, 2j+2).
 *
 * Buffer layouts (byte arrays; "row" = one storage row):
 *  - per-token row: the D/G blocks of one token and kv head;
 *  - per-channel row: D blocks (channel-ascending), each one channel over
 *    the G tokens of one token group;
 *  - main tier, contiguous: [L][batch][H_kv][capacity][row], capacity =
 *    max_T rounded up to a multiple of 32 tokens (per-token rows) or
 *    ceil(max_T/G) groups (per-channel rows);
 *  - main tier, paged (page_tokens > 0, per-token formats, W = 0):
 *    [L][n_pages][H_kv][page_tokens][row]; block_table is
 *    [batch][max_pages_per_seq] int32 (device), page of token t =
 *    block_table[seq][t / page_tokens];
 *  - hot tier when W > 0: a ring of W/G + 1 group rows (per-channel) or
 *    W + Gamma token rows (per-token); slot = index mod ring length;
 *  - cold tier: [L][batch][H_kv][capacity][row] (capacity as above);
 *  - window: [L][batch][H_kv][R + Gamma][D] 16-bit values, slot = t mod
 *    (R + Gamma).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_ARG = 1,          /* invalid argument; nothing launched */
  KVQ_ERR_UNSUPPORTED = 2,  /* valid but not implemented combination */
  KVQ_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  KVQ_ERR_CAPACITY = 4,     /* a host-visible size exceeds capacity */
  KVQ_ERR_WORKSPACE = 5     /* workspace missing or too small */
} kvq_status;

typedef enum { KVQ_DT_F16 = 0, KVQ_DT_BF16 = 1 } kvq_dtype;

/* A block spans G consecutive channels of one token (TOKEN) or one channel
 * over G consecutive tokens (CHANNEL). */
typedef enum { KVQ_AXIS_TOKEN = 0, KVQ_AXIS_CHANNEL = 1 } kvq_axis;

/* bits in {8, 4, 3, 2} (16 is accepted by the size functions only, meaning
 * plain 16-bit storage); group in {32, 128}, dividing D for TOKEN; group 32
 * for CHANNEL. */
typedef struct {
  int32_t bits;
  int32_t group;
  int32_t axis;
} kvq_fmt;

/* flags */
enum {
  KVQ_ROTATE_K = 1u << 0,  /* randomized Hadamard-128 on K before quantizing (TOKEN formats) */
  KVQ_ROTATE_V = 1u << 1,  /* the same on V */
  KVQ_K_PRE_ROPE = 1u << 2, /* K is stored pre-RoPE; decode applies split-half RoPE at position t */
  /* TBQ4 (trefon.com, "Jak 4-bitowemu cache to uchodzi: najpierw obrot"): a rotated
   * 4-bit 128-value block holds the block's L2 norm (fp16) and, per value, the index
   * of the nearest of the 16 Lloyd-Max centroids of N(0, 1/128) (see
   * kvq_tbq4_codebook).  Needs the tensor's rotation flag, 4 bits, group 128,
   * per-token blocks, one tier.  Same 66 B per 128 values.  The append kernels
   * find an index with one lookup in bins of 1/8 octave of |u|; validation
   * answers KVQ_ERR_UNSUPPORTED if two nonzero thresholds ever shared a bin
   * (the built-in table's never do). */
  KVQ_TBQ4_K = 1u << 3,
  KVQ_TBQ4_V = 1u << 4,
  /* Asymmetric blocks ("scale and zero point", nalar.dev, "Granularitas
   * kuantisasi..."): every block of that tensor (both tiers) is the fp16 scale
   * s, the fp16 zero z (the block minimum), then codes c in [0, 2^b - 1] in the
   * usual bit fields, x = c s + z: 2 more bytes per block (20 B / 32 values
   * at 4 bits, 12 B / 32 at 2 bits).  Needs 4- or 2-bit
   * blocks of 32 values, no rotation.  The tensor-core decode reads them when
   * both tensors are asymmetric (the zero adds one term per block to the
   * scores or the output); other mixes take the generic decode kernel. */
  KVQ_ZP_K = 1u << 5,
  KVQ_ZP_V = 1u << 6
};

/* Device status bits (workspace word 0), OR-ed by kernels. */
enum {
  KVQ_DEV_CAPACITY = 1u << 0, /* an append would exceed max_T, or more new tokens than max_new */
  KVQ_DEV_PAGE = 1u << 1,     /* a block_table entry outside [0, n_pages) */
  KVQ_DEV_RANGE = 1u << 2,    /* kvq_dequantize range outside [0, T) */
  KVQ_DEV_LENGTH = 1u << 3,   /* a sequence length < 0 or > max_T, or cu_new not ascending */
  KVQ_DEV_STALL = 1u << 4,    /* a decode kernel's own bulk copy into shared memory did not complete
                                 within its bounded wait; that call's outputs are undefined */
  KVQ_DEV_BOUNDS = 1u << 5    /* bounds-checked build only (libkvq_checked.so): a computed cache address
                                 fell outside its buffer segment; the access was skipped */
};

typedef struct {
  int32_t L;        /* layers held by the buffers */
  int32_t H_kv;     /* kv heads */
  int32_t H_q;      /* query heads, a multiple of H_kv, H_q/H_kv <= 8 */
  int32_t D;        /* head dim: 128 or 256 */
  int32_t batch;    /* sequences */
  int32_t max_T;    /* capacity in tokens per sequence */
  int32_t in_dtype; /* kvq_dtype of k, v, q inputs and of the window */
  kvq_fmt k_fmt, v_fmt;   /* the only tier (W = 0) or the hot tier */
  kvq_fmt k_cold, v_cold; /* cold tier when hot_window > 0 (same axis and group, fewer bits) */
  int32_t hot_window;      /* W: tokens kept in the hot tier (multiple of Gamma), 0 = one tier */
  int32_t residual_window; /* R: tokens kept in the 16-bit window, 0 allowed */
  uint32_t flags;          /* OR of KVQ_ROTATE_K, KVQ_ROTATE_V, KVQ_K_PRE_ROPE, KVQ_TBQ4_K,
                              KVQ_TBQ4_V, KVQ_ZP_K, KVQ_ZP_V (see the flags above) */
  float rope_theta;        /* RoPE base (KVQ_K_PRE_ROPE), e.g. 10000 */
  uint64_t sign_seed;      /* 0: plain Sylvester transform; else SplitMix64 sign vectors */
  int32_t page_tokens;     /* 0 = contiguous; 16 = paged main tier */
  int32_t n_pages;         /* pages in the pool (paged) */
  int32_t max_pages_per_seq; /* block_table row length (paged) */
  int32_t reserved;        /* must be 0 */
} kvq_config;

/* Every buffer is 16-byte aligned (KVQ_ERR_ARG otherwise). */
typedef struct {
  void* k_main;  /* main / hot tier of K */
  void* v_main;  /* main / hot tier of V */
  void* k_cold;  /* cold tier of K (hot_window > 0), else NULL */
  void* v_cold;  /* cold tier of V (hot_window > 0), else NULL */
  void* k_resid; /* 16-bit window of K (when R + Gamma > 1), else NULL */
  void* v_resid; /* 16-bit window of V */
  const int32_t* block_table; /* [batch][max_pages_per_seq] device (paged), else NULL */
} kvq_cache;

/* Version string of the library. */
KVQ_API const char* kvq_version(void);

/* Message of the last error returned on this thread ("" if none). */
KVQ_API const char* kvq_last_error(void);

/* Checks a configuration (the same checks every entry point makes). */
KVQ_API kvq_status kvq_validate_config(const kvq_config* cfg);

/* Bytes of one block: 2 + group*bits/8 (2*group for bits = 16)
 * (trefon.com, format table). */
KVQ_API kvq_status kvq_block_bytes(int32_t bits, int32_t group, int32_t* bytes);

/* Steady-state bytes per token over all L layers, K and V, in the format
 * that holds most of a long sequence (cold when hot_window > 0).  Scales
 * count (nalar.dev, section "Ukuran cache...": compare actual bytes per
 * token; trefon.com, section "Bajty na token"). */
KVQ_API kvq_status kvq_bytes_per_token(const kvq_config* cfg, int64_t* bytes);

/* Exact bytes the representation keeps for one sequence of T tokens over
 * all layers: cold + hot/main tiers + 16-bit window, K and V. */
KVQ_API kvq_status kvq_cache_bytes(const kvq_config* cfg, int64_t T, int64_t* bytes);

/* Bytes to allocate for the six kvq_cache buffers, in the order k_main,
 * v_main, k_cold, v_cold, k_resid, v_resid (0 = buffer not used). */
KVQ_API kvq_status kvq_buffer_sizes(const kvq_config* cfg, size_t sizes[6]);

/* Bytes of the workspace every launching call takes (status word, split
 * tickets, RoPE tables, split partials); 256-byte aligned. */
KVQ_API kvq_status kvq_workspace_bytes(const kvq_config* cfg, size_t* bytes);

/* Prepares a workspace of at least kvq_workspace_bytes: zeroes the status
 * word and tickets and fills the RoPE tables.  Call once after allocating
 * it; later calls keep the tickets at zero themselves. */
KVQ_API kvq_status kvq_workspace_init(const kvq_config* cfg, void* workspace, size_t ws_bytes, void* stream);

/* Quantize-on-append for layers [layer0, layer0 + n_layers): every new
 * token is rotated (flags), scaled per block and coded into the layout above
 * (trefon.com, format table of "Przyklad: model 27B przy 262K"; per-channel
 * keys and per-token values as troisinh.com "Tai sao Key va Value lai khac
 * nhau?"; the recent window kept unquantized as nalar.dev "Evaluasi harus
 * memisahkan...").
 *  k, v:     [n_layers][total_new][H_kv][D] in_dtype, device, 16-byte
 *            aligned (KVQ_ERR_ARG otherwise); sequences back
 *            to back in batch order (post-RoPE keys, or pre-RoPE with
 *            KVQ_K_PRE_ROPE).
 *  cu_new:   [batch + 1] int32 device, cu_new[0] = 0, cu_new[batch] =
 *            total_new; sequence b appends cu_new[b+1] - cu_new[b] tokens.
 *  seq_lens: [batch] int32 device, lengths BEFORE this append (the caller
 *            advances them after all layers, e.g. with kvq_commit_lengths).
 *  total_new, max_new: host copies of cu_new[batch] and of the largest
 *            per-sequence count (they size the grids).
 * Window tokens move into the quantized tiers by whole groups; bulk append
 * and token-by-token append give the same cache.  Inputs are finite or
 * infinite numbers; a block holding a NaN gets unspecified codes (and a NaN
 * or unspecified scale), and no other block is affected. */
KVQ_API kvq_status kvq_append(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0, int32_t n_layers,
                      const void* k, const void* v, const int32_t* cu_new, const int32_t* seq_lens,
                      int32_t total_new, int32_t max_new, void* workspace, size_t ws_bytes, void* stream);

/* seq_lens[b] += cu_new[b+1] - cu_new[b] on the device. */
KVQ_API kvq_status kvq_commit_lengths(const kvq_config* cfg, const int32_t* cu_new, int32_t* seq_lens, void* stream);

/* Decode attention of one query token per sequence, for layers
 * [layer0, layer0 + n_layers) (independent per-layer queries; n_layers > 1
 * only saves launches), read straight from the packed blocks: scores
 * s_t = q.k_t / sqrt(D) and output sum_t p_t v_t as nalar.dev "Error pada
 * key mengubah input softmax" and "Error pada value masuk setelah attention
 * probability" define them; rotated blocks are read in the rotated domain
 * (trefon.com, "Jak 4-bitowemu cache to uchodzi: najpierw obrot").
 *  q:        [n_layers][batch][H_q][D] in_dtype, device, post-RoPE.
 *  seq_lens: [batch] int32 device, tokens currently cached.
 *  out:      [n_layers][batch][H_q][D] fp32, device:
 *            out = sum_t softmax_t(q.k_t/sqrt(D)) v_t over the dequantized
 *            cache (keys RoPE-rotated at position t when stored pre-RoPE);
 *            0 for an empty sequence.
 *  num_splits: blocks per (layer, seq, kv head), 1..256; 0 picks the
 *            count (kvq_decode_splits).  With more than one, the tensor-core
 *            decode plans on the device from all lengths: when its grid is
 *            at most two waves of resident blocks, each unit of n tiles
 *            (32 tokens) is cut into ceil(n / C) nearly equal chunks for the
 *            smallest C that fits the budget, so long sequences get more
 *            blocks and short ones fewer (with a count passed here, no unit
 *            gets more than num_splits).  With 0, the budget is one whole
 *            wave of resident blocks per call where that exceeds batch x
 *            kvq_decode_splits blocks per (layer, kv head), and the grid
 *            grows to hold it (blocks past the last chunk exit at once;
 *            without room in the workspace the plain budget stays).  The
 *            result does not depend on the
 *            split beyond the order of fp32 sums.  KVQ_ERR_WORKSPACE when the
 *            workspace's partial rows cannot hold the blocks. */
KVQ_API kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0,
                                int32_t n_layers, const void* q, const int32_t* seq_lens, float* out,
                                int32_t num_splits, void* workspace, size_t ws_bytes, void* stream);

/* One decode step: appends one token to every sequence, then decode
 * attention over the cache including it (nalar.dev, "Pertumbuhan cache
 * dinamis mengubah persoalan kalibrasi": the cache grows by one entry per
 * generated token and is written online).  Equivalent to kvq_append of
 * k_new / v_new with one token per sequence followed by
 * kvq_decode_attention over seq_lens[b] + 1 tokens: the same cache bytes
 * and the same outputs.
 *  k_new, v_new: [n_layers][batch][H_kv][D] in_dtype, device, 16-byte
 *            aligned: the new token of every (layer, sequence).
 *  q, out, num_splits: as kvq_decode_attention.
 *  seq_lens: [batch] int32 device, lengths BEFORE the step; the new token
 *            is at position seq_lens[b].  Not advanced here: the caller
 *            advances them after all layers (kvq_commit_lengths with
 *            cu_new = 0, 1, ..., batch).
 * When the tensor-core decode handles the formats the step is one launch:
 * the blocks that own the (at most three) tiles the token changes -- its
 * window slot, the unit leaving the window, the group leaving the hot tier
 * -- write them and then decode them; no block waits for another.  Other
 * formats run the append and decode launches in turn. */
KVQ_API kvq_status kvq_decode_step(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0, int32_t n_layers,
                                   const void* k_new, const void* v_new, const void* q, const int32_t* seq_lens,
                                   float* out, int32_t num_splits, void* workspace, size_t ws_bytes, void* stream);

/* Kernel launches one kvq_decode_step call makes (1 when fused). */
KVQ_API kvq_status kvq_step_launches(const kvq_config* cfg, int32_t* launches);

/* The split count per (layer, seq, kv head) kvq_decode_attention takes for
 * num_splits = 0: the count with the best fill of whole waves of resident
 * blocks (the device's SM count), each block keeping at least 8 tiles of the
 * longest possible sequence (48 for rotated formats).  A call whose chunks
 * are planned on the device may widen it to give the plan one whole wave
 * (kvq_decode_attention). */
KVQ_API kvq_status kvq_decode_splits(const kvq_config* cfg, int32_t n_layers, int32_t* splits);

/* Dequantizes tokens [t0, t1) of (layer, seq) to fp32 k_out, v_out
 * [t1 - t0][H_kv][D] (device) in the original domain: x = code * scale
 * (+ zero) per block (trefon.com, format table), rotation undone, keys as
 * stored (pre-RoPE when flagged).  k_out and v_out hold at least
 * (t1 - t0) * H_kv * D floats each; the caller owns them.  seq_lens as for decode; a range beyond
 * the current length sets KVQ_DEV_RANGE and writes nothing. */
KVQ_API kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_cache* cache, int32_t layer, int32_t seq,
                          int32_t t0, int32_t t1, const int32_t* seq_lens, float* k_out, float* v_out,
                          void* workspace, size_t ws_bytes, void* stream);

/* Size of the library's built-in device scratch used by
 * kvq_decode_attention_static (32 MiB on every GPU that loads the library,
 * held until the process exits). */
#define KVQ_STATIC_SCRATCH_BYTES (32u << 20)

/* Decode attention that allocates nothing and takes no workspace.
 *
 * There is no counterpart on the pages: this is an addition of this library
 * for callers that cannot hand it device memory.  Examples are code whose
 * device memory all belongs to another runtime's pool that it may not
 * allocate from, and plugins that are given inputs and outputs but no
 * scratch buffer.  kvq_decode_attention needs the caller to allocate a
 * workspace; this variant keeps the same scratch (split partials, tickets,
 * status word, RoPE tables) in a fixed device array inside the library.
 *
 * Arguments and results are those of kvq_decode_attention without the
 * workspace.  The call needs 256 B + 4 B per (layer, sequence, kv head)
 * unit + the RoPE tables (KVQ_K_PRE_ROPE) + the split partials; a call that
 * needs more than KVQ_STATIC_SCRATCH_BYTES returns KVQ_ERR_WORKSPACE and
 * launches nothing (pass a smaller n_layers or num_splits).  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on each device looks up the array's device address with
 * that device current, so make that first call before any stream capture.
 * Every call on a device uses the same array and leaves its contents
 * behind; each call clears the parts that must start at zero (tickets and
 * status word) on `stream`, so calls that overlap on the GPU (two streams,
 * or two threads) race and must be serialized by the caller.  Device status
 * bits of these calls are not reported. */
KVQ_API kvq_status kvq_decode_attention_static(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0,
                                               int32_t n_layers, const void* q, const int32_t* seq_lens,
                                               float* out, int32_t num_splits, void* stream);

/* Kernel launches one kvq_append call (with new tokens) and one
 * kvq_decode_attention call make for this configuration, e.g. to budget
 * launches per decode step.  No pages counterpart: library bookkeeping. */
KVQ_API kvq_status kvq_launch_counts(const kvq_config* cfg, int32_t* append_launches, int32_t* decode_launches);

/* The TBQ4 tables the library uses: the 16 Lloyd-Max centroids of
 * N(0, sigma^2), sigma = 1/sqrt(128), ascending, from Lloyd's algorithm run
 * on the host in fp64 and rounded once to fp16 (the lookup table), and the
 * 15 decision thresholds, the exact midpoints of neighbouring entries.  A
 * value u = y / norm (fp32, y the rotated value) takes the index of the
 * number of thresholds strictly below u; it decodes as centroid[index] *
 * norm.  The norm is fp16(min(sqrt(S), 65504)) with S = (p0 + p1) + (p2 + p3)
 * in fp32, p_k the sum of y_i^2 over the k-th run of 32 values in index
 * order.  No device work; the tables are computed once per process. */
KVQ_API kvq_status kvq_tbq4_codebook(float centroids[16], float thresholds[15]);

/* Testing hook of the failure-detection path; no counterpart on the pages.
 * While polls > 0, every tensor-core decode launch (kvq_decode_attention,
 * kvq_decode_step, kvq_decode_attention_static) makes its warps' first copy
 * wait on a shared-memory barrier that nothing ever completes, bounded by
 * `polls` polls: the wait runs out, KVQ_DEV_STALL is set, the warp waits
 * (with the normal bound) for its bulk copies still in flight and the
 * kernel finishes; that call's outputs are undefined.  polls = 0 (the
 * default) turns it off.  Process-wide; polls outside [0, 2^20] give
 * KVQ_ERR_ARG.  Not for production use. */
KVQ_API kvq_status kvq_test_force_stall(int32_t polls);

/* Testing hook of the bounds-checked build (libkvq_checked.so, compiled
 * with KVQ_BOUNDS_CHECK); no counterpart on the pages.  Later calls treat
 * the last `rows` rows (or page rows) of every cache segment as outside the
 * buffer, so accesses there set KVQ_DEV_BOUNDS and are skipped: a test that
 * the checks fire without any real out-of-bounds access.  0 (the default)
 * turns it off.  The normal build answers KVQ_ERR_UNSUPPORTED for rows > 0. */
KVQ_API kvq_status kvq_test_shrink_bounds(int32_t rows);

/* Synchronizes `stream` and reads the device status word (KVQ_DEV_* bits). */
KVQ_API kvq_status kvq_read_device_status(const void* workspace, uint32_t* bits, void* stream);

/* Clears the device status word. */
KVQ_API kvq_status kvq_clear_device_status(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
