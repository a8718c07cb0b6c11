// Internal definitions shared by the libkvq translation units: the derived
// cache layout (POD, passed to kernels by value), tier arithmetic and
// address helpers.  Everything here follows the contract stated in kvq.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/kvq.h"

#define KVQ_HD __host__ __device__ __forceinline__

namespace kvq {

constexpr int kTile = 32;        // tokens per decode / append tile
constexpr int kMaxGqa = 8;       // query heads per kv head
constexpr int kTargetCtas = 608; // 4 x 152 SMs: split heuristic target
constexpr int kMaxSplits = 256;
// Split partials merge in groups of kCombineFan consecutive chunks, then the
// group rows: tickets per unit are one for the unit and one per group.
constexpr int kCombineFan = 8;
constexpr int kTicketsPerUnit = 1 + kMaxSplits / kCombineFan;
constexpr size_t kWsAlign = 256;
// float2 rows of D/2 after the base rows of the RoPE tables: the plain
// offsets, the offsets in the lanes' order, the fp16 hi / lo turn table
constexpr int kRopeExtraRows = 3 * kTile;

struct FmtInfo {
  int bits;   // 8, 4, 3, 2 (0 = unused)
  int group;  // G
  int axis;   // KVQ_AXIS_*
  int bb;     // block bytes
  int qmax;   // 2^(bits-1) - 1
  int row;    // bytes of one storage row
  int codebook;  // 1: TBQ4 blocks (fp16 L2 norm + Lloyd-Max centroid indices)
  int zp;        // 1: asymmetric blocks (fp16 scale, fp16 zero, codes 0..2^b-1)
};

// Everything a kernel needs to find a byte of the cache.
struct Layout {
  int L, B, H, Hq, D, g;
  int max_T;
  int dtype;
  int gam;         // Gamma: token granularity of quantization
  int R;           // 16-bit window
  int W;           // hot window (0 = one tier)
  int ring;        // window ring slots (0 = none)
  int tiered, paged;
  int pt, n_pages, max_pages;
  uint32_t flags;
  float theta;
  uint32_t d1[4], d2[4];  // Hadamard sign masks (bit set = -1)
  FmtInfo kf, vf, kc, vc;
  int64_t rows_k_main, rows_v_main;  // rows per (layer, seq, head) of the main tier (contiguous / ring)
  int64_t rows_k_cold, rows_v_cold;
  int hot_ring_k, hot_ring_v;        // ring length of the hot tier (rows) when tiered
  float cb[16];                      // TBQ4 centroid table (fp16 values, ascending), when used
  float cbt[15];                     // TBQ4 decision thresholds
  int bounds_shrink;                 // bounds-checked build: rows taken off every segment's limit (tests)
};

struct CachePtrs {
  uint8_t* k_main;
  uint8_t* v_main;
  uint8_t* k_cold;
  uint8_t* v_cold;
  uint16_t* k_resid;
  uint16_t* v_resid;
  const int32_t* block_table;
  uint32_t* status;  // device status word (the bounds-checked build records misses there)
};

// Workspace layout offsets (bytes).
struct WsLayout {
  size_t status;    // uint32 status word
  size_t tickets;   // uint32 per decode unit
  size_t rope;      // float2 base[n_base][D/2], off[kTile][D/2], off in lane order (kTile x D/2),
                    // then the fp16 hi / lo turn table (kTile x D/2 float2 of space)
  size_t partials;  // float per (unit, split): g * part_row(D)
  size_t total;
  int max_units;
  int max_partials;  // unit-split pairs
  int rope_base_rows;
};

KVQ_HD int qmax_of(int bits) { return (1 << (bits - 1)) - 1; }

KVQ_HD int block_bytes_of(int bits, int group) {
  return bits == 16 ? 2 * group : 2 + group * bits / 8;
}

// ---- tier arithmetic ------------------------------------------------------

// Gamma is 1 or 32 (per-channel groups are 32 tokens), so rounding down to a
// multiple of Gamma is a mask.
KVQ_HD int q_end_of(const Layout& lo, int T) {
  if (T <= lo.R) return 0;
  return (T - lo.R) & ~(lo.gam - 1);
}

KVQ_HD int c_end_of(const Layout& lo, int T) {
  if (lo.W <= 0) return 0;
  int qe = q_end_of(lo, T);
  if (qe <= lo.W) return 0;
  return (qe - lo.W) & ~(lo.gam - 1);
}

// ---- addresses --------------------------------------------------------------

// Bounds-checked build (-DKVQ_BOUNDS_CHECK, a stand-in for a memory checker):
// every row helper checks its indices against the buffer's dimensions
// (layer, sequence, kv head, row or page of the segment); a miss sets
// KVQ_DEV_BOUNDS and yields row 0 of the buffer, so nothing outside the
// caller's buffers is touched.  Sites that move several rows from one row
// pointer check the run with span_ok.  The normal build compiles none of it.
#if defined(KVQ_BOUNDS_CHECK) && defined(__CUDA_ARCH__)
__device__ __forceinline__ bool kvq_bound(const CachePtrs& cp, bool ok) {
  if (!ok && cp.status) atomicOr(cp.status, KVQ_DEV_BOUNDS);
  return ok;
}
#define KVQ_CHECK(cond) kvq_bound(cp, (cond))
#else
#define KVQ_CHECK(cond) true
#endif

KVQ_HD const FmtInfo& fmt_main(const Layout& lo, int which) { return which ? lo.vf : lo.kf; }
KVQ_HD const FmtInfo& fmt_cold(const Layout& lo, int which) { return which ? lo.vc : lo.kc; }

// Main-tier row holding token t (per-token) or group t/G (per-channel);
// nullptr (and *bad set) for a page id out of range.
KVQ_HD uint8_t* main_row(const Layout& lo, const CachePtrs& cp, int which, int layer, int seq, int h,
                         int t, bool* bad) {
  const FmtInfo& f = fmt_main(lo, which);
  uint8_t* base = which ? cp.v_main : cp.k_main;
  if (lo.paged) {
    if (!KVQ_CHECK(seq >= 0 && seq < lo.B && t >= 0 && t / lo.pt < lo.max_pages)) return base;
    int page = cp.block_table[(int64_t)seq * lo.max_pages + t / lo.pt];
    if (page < 0 || page >= lo.n_pages) {
      *bad = true;
      return nullptr;
    }
    if (!KVQ_CHECK(layer >= 0 && layer < lo.L && h >= 0 && h < lo.H && t % lo.pt < lo.pt - lo.bounds_shrink))
      return base;
    int64_t idx = (((int64_t)layer * lo.n_pages + page) * lo.H + h) * lo.pt + (t % lo.pt);
    return base + idx * f.row;
  }
  int64_t rows = which ? lo.rows_v_main : lo.rows_k_main;
  int64_t r;
  if (f.axis == KVQ_AXIS_CHANNEL) {
    int gi = t / f.group;
    r = lo.tiered ? (gi % (which ? lo.hot_ring_v : lo.hot_ring_k)) : gi;
  } else {
    r = lo.tiered ? (t % (which ? lo.hot_ring_v : lo.hot_ring_k)) : t;
  }
  if (!KVQ_CHECK(layer >= 0 && layer < lo.L && seq >= 0 && seq < lo.B && h >= 0 && h < lo.H && t >= 0 &&
                 r < rows - lo.bounds_shrink))
    return base;
  int64_t idx = (((int64_t)layer * lo.B + seq) * lo.H + h) * rows + r;
  return base + idx * f.row;
}

KVQ_HD uint8_t* cold_row(const Layout& lo, const CachePtrs& cp, int which, int layer, int seq, int h, int t) {
  const FmtInfo& f = fmt_cold(lo, which);
  uint8_t* base = which ? cp.v_cold : cp.k_cold;
  int64_t rows = which ? lo.rows_v_cold : lo.rows_k_cold;
  int64_t r = (f.axis == KVQ_AXIS_CHANNEL) ? t / f.group : t;
  if (!KVQ_CHECK(layer >= 0 && layer < lo.L && seq >= 0 && seq < lo.B && h >= 0 && h < lo.H && t >= 0 &&
                 r < rows - lo.bounds_shrink))
    return base;
  int64_t idx = (((int64_t)layer * lo.B + seq) * lo.H + h) * rows + r;
  return base + idx * f.row;
}

KVQ_HD uint16_t* resid_row(const Layout& lo, const CachePtrs& cp, int which, int layer, int seq, int h, int t) {
  uint16_t* base = which ? cp.v_resid : cp.k_resid;
  if (!KVQ_CHECK(layer >= 0 && layer < lo.L && seq >= 0 && seq < lo.B && h >= 0 && h < lo.H && t >= 0 &&
                 t % lo.ring < lo.ring - lo.bounds_shrink))
    return base;
  int64_t idx = (((int64_t)layer * lo.B + seq) * lo.H + h) * lo.ring + (t % lo.ring);
  return base + idx * lo.D;
}

// Whether [p, p + bytes) lies inside one segment of cache buffer `buf` (0
// k_main, 1 v_main, 2 k_cold, 3 v_cold): the rows of one (layer, sequence, kv
// head), or of one page and kv head when paged.  Always true in the normal
// build; in the bounds-checked build a miss sets KVQ_DEV_BOUNDS.
KVQ_HD bool span_ok(const Layout& lo, const CachePtrs& cp, int buf, const void* p, int64_t bytes) {
#if defined(KVQ_BOUNDS_CHECK) && defined(__CUDA_ARCH__)
  const bool cold = buf >= 2;
  const int which = buf & 1;
  const FmtInfo& f = cold ? fmt_cold(lo, which) : fmt_main(lo, which);
  const uint8_t* base = cold ? (which ? cp.v_cold : cp.k_cold) : (which ? cp.v_main : cp.k_main);
  int64_t rows, n_seg;
  if (!cold && lo.paged) {
    rows = lo.pt;
    n_seg = (int64_t)lo.L * lo.n_pages * lo.H;
  } else {
    rows = cold ? (which ? lo.rows_v_cold : lo.rows_k_cold) : (which ? lo.rows_v_main : lo.rows_k_main);
    n_seg = (int64_t)lo.L * lo.B * lo.H;
  }
  const int64_t seg_bytes = rows * f.row;
  const int64_t off = reinterpret_cast<const uint8_t*>(p) - base;
  const int64_t seg = off >= 0 ? off / seg_bytes : -1;
  return kvq_bound(cp, bytes >= 0 && seg >= 0 && seg < n_seg &&
                           off + bytes <= seg * seg_bytes + (rows - lo.bounds_shrink) * f.row);
#else
  (void)lo;
  (void)cp;
  (void)buf;
  (void)p;
  (void)bytes;
  return true;
#endif
}

// ---- number helpers -----------------------------------------------------------

__device__ __forceinline__ float in_to_f32(uint16_t bits, int dtype) {
  if (dtype == KVQ_DT_F16) return __half2float(__ushort_as_half(bits));
  return __uint_as_float(((uint32_t)bits) << 16);
}

__device__ __forceinline__ float sign_of(const uint32_t* mask, int i) {
  return ((mask[i >> 5] >> (i & 31)) & 1u) ? -1.0f : 1.0f;
}

// TBQ4 tables (host, computed once): 16 centroids, 15 thresholds, fp32.
void tbq4_tables(float* centroids, float* thresholds);
bool tbq4_bins_ok();

// ---- programmatic dependent launch -------------------------------------------
// Decode kernels are launched with programmatic stream serialization: the
// stream's next kernel may launch while this one drains, and every such
// kernel first waits (griddepcontrol.wait) for the previous grid of the
// stream to complete with its memory visible, so the order of effects is the
// plain stream order.  Consecutive decode calls then overlap one grid's tail
// with the next one's block launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::); }

template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- launchers (defined in the kernel translation units) -------------------

struct AppendArgs {
  Layout lo;
  CachePtrs cp;
  int layer0, n_layers;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* cu_new;
  const int32_t* seq_lens;
  int total_new, max_new;
  uint32_t* status;
  int one_per_seq;  // 1: one new token per sequence, row `seq` of k / v (cu_new unused)
};

struct DecodeArgs {
  Layout lo;
  CachePtrs cp;
  int layer0, n_layers;
  const uint16_t* q;
  const int32_t* seq_lens;
  float* out;
  int splits;        // blocks per (layer, sequence, kv head) in the grid
  int budget;        // chunk plan: blocks per (layer, kv head) it may use (at most batch x splits)
  int min_chunk;     // tensor-core decode: least tiles per chunk of a unit
  int fixed_splits;  // 1: the caller fixed `splits`, so no unit is cut into more chunks
  int chunked;       // 1: plan chunks by tile count; 0: split every unit evenly
  uint32_t* status;
  uint32_t* tickets;
  float* partials;
  const float2* rope;  // base rows then offsets
  int rope_base_rows;
  int len_add;      // the attended length is seq_lens[b] + len_add (1 in a decode step)
  int stall_polls;  // > 0: failure-detection test mode (kvq_test_force_stall)
  AppendArgs step;  // fused decode step: the append of the new token (step.k == nullptr otherwise)
};

struct DequantArgs {
  Layout lo;
  CachePtrs cp;
  int layer, seq, t0, t1;
  const int32_t* seq_lens;
  float* k_out;
  float* v_out;
  uint32_t* status;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
// Specialized phase B (quantize) of an append when one exists for both
// tensors' formats; false when nothing was launched.
bool launch_fast_quantize(const AppendArgs& a, cudaStream_t s);
bool fast_quantize_available(const AppendArgs& a);
cudaError_t launch_commit_lengths(const int32_t* cu_new, int32_t* seq_lens, int batch, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);  // tensor-core path when it fits, else generic
cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s);
// Fused decode step (a.step holds the append of one token per sequence, a.len_add = 1): one tensor-core
// launch into *err unless `dry`; false when the formats take the generic path.
bool launch_decode_step_fused(const DecodeArgs& a, cudaStream_t s, bool dry, cudaError_t* err);
cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_rope_tables(float2* rope, int base_rows, int D, float theta, cudaStream_t s);

}  // namespace kvq
