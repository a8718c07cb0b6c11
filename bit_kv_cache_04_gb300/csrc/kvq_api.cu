// Host side of the C ABI declared in include/kvq.h: argument validation,
// the size law, buffer and workspace sizing, and kernel launches.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "kvq_internal.cuh"
#include "split_combine.cuh"
#include "tbq4_bins.cuh"

using namespace kvq;

namespace {

// Rows taken off every cache segment's limit in the bounds-checked build
// (kvq_test_shrink_bounds); read by make_layout.
std::atomic<int> g_bounds_shrink{0};

thread_local std::string g_last_error;

kvq_status fail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvq_status ok() {
  g_last_error.clear();
  return KVQ_OK;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_bits(int bits, bool allow16) { return bits == 8 || bits == 4 || bits == 3 || bits == 2 || (allow16 && bits == 16); }

kvq_status check_fmt(const kvq_fmt& f, int D, const char* name, bool allow16) {
  if (!valid_bits(f.bits, allow16)) return fail(KVQ_ERR_ARG, "%s.bits=%d not in {8,4,3,2}", name, f.bits);
  if (f.axis != KVQ_AXIS_TOKEN && f.axis != KVQ_AXIS_CHANNEL) return fail(KVQ_ERR_ARG, "%s.axis=%d", name, f.axis);
  if (f.group != 32 && f.group != 128) return fail(KVQ_ERR_ARG, "%s.group=%d not in {32,128}", name, f.group);
  if (f.axis == KVQ_AXIS_TOKEN && D % f.group != 0) return fail(KVQ_ERR_ARG, "%s.group=%d does not divide D=%d", name, f.group, D);
  if (f.axis == KVQ_AXIS_CHANNEL && f.group != 32) return fail(KVQ_ERR_UNSUPPORTED, "%s: per-channel groups are 32 tokens", name);
  if (f.bits == 16 && f.axis != KVQ_AXIS_TOKEN) return fail(KVQ_ERR_ARG, "%s: 16-bit storage is per-token", name);
  return KVQ_OK;
}

// Checks shared by all entry points. allow16: size-law-only formats.
kvq_status check_config(const kvq_config* c, bool allow16) {
  if (!c) return fail(KVQ_ERR_ARG, "config is NULL");
  if (c->reserved != 0) return fail(KVQ_ERR_ARG, "reserved must be 0");
  if (c->L < 1 || c->H_kv < 1 || c->H_q < 1 || c->batch < 1 || c->max_T < 1)
    return fail(KVQ_ERR_ARG, "L, H_kv, H_q, batch, max_T must be >= 1");
  if (c->H_q % c->H_kv != 0) return fail(KVQ_ERR_ARG, "H_q=%d is not a multiple of H_kv=%d", c->H_q, c->H_kv);
  if (c->H_q / c->H_kv > kMaxGqa) return fail(KVQ_ERR_UNSUPPORTED, "H_q/H_kv=%d > %d", c->H_q / c->H_kv, kMaxGqa);
  if (c->D != 128 && c->D != 256) return fail(KVQ_ERR_UNSUPPORTED, "D=%d not in {128,256}", c->D);
  if (c->in_dtype != KVQ_DT_F16 && c->in_dtype != KVQ_DT_BF16) return fail(KVQ_ERR_ARG, "in_dtype=%d", c->in_dtype);
  kvq_status st;
  if ((st = check_fmt(c->k_fmt, c->D, "k_fmt", allow16)) != KVQ_OK) return st;
  if ((st = check_fmt(c->v_fmt, c->D, "v_fmt", allow16)) != KVQ_OK) return st;
  if (c->hot_window < 0 || c->residual_window < 0) return fail(KVQ_ERR_ARG, "negative window");
  int gam = 1;
  if (c->k_fmt.axis == KVQ_AXIS_CHANNEL) gam = c->k_fmt.group;
  if (c->v_fmt.axis == KVQ_AXIS_CHANNEL) gam = c->v_fmt.group;
  if (c->hot_window > 0) {
    if ((st = check_fmt(c->k_cold, c->D, "k_cold", allow16)) != KVQ_OK) return st;
    if ((st = check_fmt(c->v_cold, c->D, "v_cold", allow16)) != KVQ_OK) return st;
    if (c->k_cold.axis != c->k_fmt.axis || c->k_cold.group != c->k_fmt.group ||
        c->v_cold.axis != c->v_fmt.axis || c->v_cold.group != c->v_fmt.group)
      return fail(KVQ_ERR_UNSUPPORTED, "cold formats must keep the hot formats' axis and group");
    if (gam == 1) return fail(KVQ_ERR_UNSUPPORTED, "hot/cold tiers need a per-channel (token-group) format");
    if (c->hot_window % gam != 0) return fail(KVQ_ERR_ARG, "hot_window=%d not a multiple of %d", c->hot_window, gam);
  }
  uint32_t known = KVQ_ROTATE_K | KVQ_ROTATE_V | KVQ_K_PRE_ROPE | KVQ_TBQ4_K | KVQ_TBQ4_V | KVQ_ZP_K | KVQ_ZP_V;
  if (c->flags & ~known) return fail(KVQ_ERR_ARG, "unknown flags 0x%x", c->flags & ~known);
  if ((c->flags & KVQ_ROTATE_K) && c->k_fmt.axis != KVQ_AXIS_TOKEN)
    return fail(KVQ_ERR_UNSUPPORTED, "rotation needs per-token K blocks");
  if ((c->flags & KVQ_ROTATE_V) && c->v_fmt.axis != KVQ_AXIS_TOKEN)
    return fail(KVQ_ERR_UNSUPPORTED, "rotation needs per-token V blocks");
  if ((c->flags & KVQ_ROTATE_K) && (c->flags & KVQ_K_PRE_ROPE))
    return fail(KVQ_ERR_UNSUPPORTED, "pre-RoPE keys with rotated K: RoPE pairs do not commute with the transform");
  if ((c->flags & KVQ_K_PRE_ROPE) && !(c->rope_theta > 1.0f)) return fail(KVQ_ERR_ARG, "rope_theta must be > 1");
  for (int t = 0; t < 2; ++t) {
    const uint32_t zb = t ? KVQ_ZP_V : KVQ_ZP_K, rz = t ? KVQ_ROTATE_V : KVQ_ROTATE_K;
    if (!(c->flags & zb)) continue;
    const kvq_fmt& f = t ? c->v_fmt : c->k_fmt;
    const kvq_fmt& fc = t ? c->v_cold : c->k_cold;
    auto zp_ok = [](const kvq_fmt& x) { return (x.bits == 4 || x.bits == 2) && x.group == 32; };
    if ((c->flags & rz) || !zp_ok(f) || (c->hot_window > 0 && !zp_ok(fc)))
      return fail(KVQ_ERR_UNSUPPORTED, "zero-point blocks need 4- or 2-bit blocks of 32 values and no rotation");
  }
  for (int t = 0; t < 2; ++t) {
    const uint32_t tb = t ? KVQ_TBQ4_V : KVQ_TBQ4_K, rb = t ? KVQ_ROTATE_V : KVQ_ROTATE_K;
    const kvq_fmt& f = t ? c->v_fmt : c->k_fmt;
    if (!(c->flags & tb)) continue;
    if (!(c->flags & rb) || f.bits != 4 || f.group != 128 || f.axis != KVQ_AXIS_TOKEN || c->hot_window > 0)
      return fail(KVQ_ERR_UNSUPPORTED, "TBQ4 needs the rotation, 4-bit per-token blocks of 128 and one tier");
    if (!kvq::tbq4_bins_ok())
      return fail(KVQ_ERR_UNSUPPORTED, "TBQ4 midpoints too close for the binned index lookup");
  }
  if (c->page_tokens < 0) return fail(KVQ_ERR_ARG, "page_tokens < 0");
  if (c->page_tokens > 0) {
    if (c->k_fmt.axis != KVQ_AXIS_TOKEN || c->v_fmt.axis != KVQ_AXIS_TOKEN || c->hot_window > 0)
      return fail(KVQ_ERR_UNSUPPORTED, "paging needs per-token formats and one tier");
    if (c->n_pages < 1) return fail(KVQ_ERR_ARG, "n_pages < 1");
    if ((int64_t)c->max_pages_per_seq * c->page_tokens < c->max_T)
      return fail(KVQ_ERR_ARG, "max_pages_per_seq * page_tokens < max_T");
  }
  return KVQ_OK;
}

FmtInfo make_fmt(const kvq_fmt& f, int D, bool codebook = false, bool zp = false) {
  FmtInfo r{};
  r.codebook = codebook ? 1 : 0;
  r.zp = zp ? 1 : 0;
  if (f.bits == 0) return r;
  r.bits = f.bits;
  r.group = f.group;
  r.axis = f.axis;
  r.bb = block_bytes_of(f.bits, f.group) + (zp ? 2 : 0);
  r.qmax = f.bits == 16 ? 0 : qmax_of(f.bits);
  r.row = f.axis == KVQ_AXIS_TOKEN ? (D / f.group) * r.bb : D * r.bb;
  return r;
}

// Lloyd's algorithm (S. P. Lloyd 1982; J. Max 1960) for the 16-point
// minimum-MSE quantizer of N(0, sigma^2), sigma = 1/sqrt(128), in double:
// thresholds at the midpoints of neighbouring centroids, centroids at the
// conditional means E[Z | a < Z < b] = (pdf(a) - pdf(b)) / (Q(a) - Q(b)) with
// Q the upper tail, iterated on the positive half (the density is symmetric)
// until no centroid moves by more than 1e-15 sigma.
void lloyd_max_normal16(double* centroids) {
  const double inv_sqrt2pi = 0.3989422804014327, inv_sqrt2 = 0.7071067811865476;
  auto pdf = [&](double z) { return inv_sqrt2pi * std::exp(-0.5 * z * z); };
  auto upper = [&](double z) { return 0.5 * std::erfc(z * inv_sqrt2); };
  double c[8];
  for (int j = 0; j < 8; ++j) c[j] = 0.5 * (j + 0.5);
  for (int it = 0; it < 100000; ++it) {
    double t[9];
    t[0] = 0.0;
    for (int j = 1; j < 8; ++j) t[j] = 0.5 * (c[j - 1] + c[j]);
    double moved = 0.0;
    double nc[8];
    for (int j = 0; j < 8; ++j) {
      const double a = t[j];
      const double pb = j + 1 < 8 ? pdf(t[j + 1]) : 0.0, qb = j + 1 < 8 ? upper(t[j + 1]) : 0.0;
      nc[j] = (pdf(a) - pb) / (upper(a) - qb);
      moved = std::max(moved, std::fabs(nc[j] - c[j]));
    }
    for (int j = 0; j < 8; ++j) c[j] = nc[j];
    if (moved <= 1e-15) break;
  }
  const double sigma = 1.0 / std::sqrt(128.0);
  for (int j = 0; j < 8; ++j) {
    centroids[8 + j] = c[j] * sigma;
    centroids[7 - j] = -c[j] * sigma;
  }
}

uint64_t splitmix64_next(uint64_t* state) {
  // SplitMix64 (Steele, Lea and Flood, 2014).
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

Layout make_layout(const kvq_config* c) {
  Layout lo{};
  lo.L = c->L;
  lo.B = c->batch;
  lo.H = c->H_kv;
  lo.Hq = c->H_q;
  lo.D = c->D;
  lo.g = c->H_q / c->H_kv;
  lo.max_T = c->max_T;
  lo.dtype = c->in_dtype;
  lo.gam = 1;
  if (c->k_fmt.axis == KVQ_AXIS_CHANNEL) lo.gam = c->k_fmt.group;
  if (c->v_fmt.axis == KVQ_AXIS_CHANNEL) lo.gam = c->v_fmt.group;
  lo.R = c->residual_window;
  lo.W = c->hot_window;
  lo.ring = (lo.R == 0 && lo.gam == 1) ? 0 : lo.R + lo.gam;
  lo.tiered = c->hot_window > 0;
  lo.paged = c->page_tokens > 0;
  lo.pt = c->page_tokens;
  lo.n_pages = c->n_pages;
  lo.max_pages = c->max_pages_per_seq;
  lo.flags = c->flags;
  lo.theta = c->rope_theta;
  lo.bounds_shrink = g_bounds_shrink.load();
  if (c->sign_seed != 0) {
    uint64_t st = c->sign_seed, w[4];
    for (int i = 0; i < 4; ++i) w[i] = splitmix64_next(&st);
    for (int j = 0; j < 4; ++j) {
      lo.d1[j] = (uint32_t)(w[j / 2] >> (32 * (j % 2)));
      lo.d2[j] = (uint32_t)(w[2 + j / 2] >> (32 * (j % 2)));
    }
  }
  const bool zk = (c->flags & KVQ_ZP_K) != 0, zv = (c->flags & KVQ_ZP_V) != 0;
  lo.kf = make_fmt(c->k_fmt, c->D, (c->flags & KVQ_TBQ4_K) != 0, zk);
  lo.vf = make_fmt(c->v_fmt, c->D, (c->flags & KVQ_TBQ4_V) != 0, zv);
  if (c->flags & (KVQ_TBQ4_K | KVQ_TBQ4_V)) tbq4_tables(lo.cb, lo.cbt);
  if (lo.tiered) {
    lo.kc = make_fmt(c->k_cold, c->D, false, zk);
    lo.vc = make_fmt(c->v_cold, c->D, false, zv);
  }
  // per-token capacity is rounded up to whole 32-token tiles so that every
  // tile starts 16-byte aligned and lies inside the buffer
  auto rows_abs = [&](const FmtInfo& f) -> int64_t {
    return f.axis == KVQ_AXIS_TOKEN ? (int64_t)((c->max_T + kTile - 1) / kTile * kTile)
                                    : (int64_t)((c->max_T + f.group - 1) / f.group);
  };
  auto rows_ring = [&](const FmtInfo& f) -> int {
    return f.axis == KVQ_AXIS_TOKEN ? c->hot_window + lo.gam : c->hot_window / f.group + 1;
  };
  if (lo.tiered) {
    lo.hot_ring_k = rows_ring(lo.kf);
    lo.hot_ring_v = rows_ring(lo.vf);
    lo.rows_k_main = lo.hot_ring_k;
    lo.rows_v_main = lo.hot_ring_v;
    lo.rows_k_cold = rows_abs(lo.kc);
    lo.rows_v_cold = rows_abs(lo.vc);
  } else {
    lo.rows_k_main = rows_abs(lo.kf);
    lo.rows_v_main = rows_abs(lo.vf);
  }
  return lo;
}

int64_t fmt_bytes(const kvq_fmt& f, int64_t n_tokens, int D, bool zp) {
  int64_t bb = block_bytes_of(f.bits, f.group) + (zp ? 2 : 0);
  if (f.axis == KVQ_AXIS_TOKEN) return n_tokens * (D / f.group) * bb;
  return (n_tokens / f.group) * D * bb;
}

// Streaming multiprocessors of the current device, read once per device
// from its attributes.  Without a usable device (host-only sizing queries)
// the count of a GB300 (152) stands in, so sizes stay deterministic there.
int sm_count() {
  constexpr int kMaxDev = 64, kDefaultSms = 152;
  static std::mutex mu;
  static int cached[kMaxDev] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    (void)cudaGetLastError();
    return kDefaultSms;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = kDefaultSms;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Token splits per (layer, sequence, kv head): the count whose grid fills
// whole waves of resident CTAs best (SMs x 4 CTAs for D = 128, x 2 for
// D = 256), with at least 8 tiles per split and no more growth once the grid
// holds 8 waves.
constexpr int64_t kMinTilesPerSplit = 8, kMinTilesPerSplitRotated = 48;
// The least tiles per chunk when the device plans chunks (rotated layouts):
// with the one-wave budget a ragged batch of 2K-8K-token sequences decoded
// per layer took 1.12 ms with a floor of 16, 24 or 32 tiles, 1.28 ms with 48.
constexpr int kMinChunkRotated = 32;

int splits_for(const kvq_config* c, int n_layers) {
  const int64_t units = (int64_t)n_layers * c->batch * c->H_kv;
  const int64_t tiles = (c->max_T + kTile - 1) / kTile + 2;
  const int64_t resident = (int64_t)sm_count() * (c->D == 128 ? 4 : 2);
  // every split keeps at least a minimum of tiles of capacity.  Rotated
  // layouts set a higher one: their per-block setup also rotates the query
  // and un-rotates the output (a ragged batch of 2K-8K-token sequences
  // decoded per layer took 2.15 ms with 19 splits per unit, 1.53 ms with 4;
  // unrotated 1K-token layouts run faster with small splits)
  const bool rotated = (c->flags & (KVQ_ROTATE_K | KVQ_ROTATE_V)) != 0;
  int64_t cap = tiles / (rotated ? kMinTilesPerSplitRotated : kMinTilesPerSplit);
  if (cap < 1) cap = 1;
  if (cap > kMaxSplits) cap = kMaxSplits;
  int best = 1;
  double best_eff = -1.0;
  for (int64_t sp = 1; sp <= cap; ++sp) {
    const int64_t ctas = units * sp;
    const int64_t waves = (ctas + resident - 1) / resident;
    const double eff = (double)ctas / (double)(waves * resident);
    if (eff > best_eff + 1e-9) {
      best = (int)sp;
      best_eff = eff;
    }
    if (ctas >= 8 * resident) break;
  }
  return best;
}

// The grid and chunking of a decode call (see plan_work): the grid's blocks
// per (layer, sequence, kv head) `*splits` (the caller's count, else
// splits_for), the least tiles per chunk, whether the caller fixed the split
// count, whether to plan chunks by tile count at all (grids of up to two
// waves of resident blocks; larger grids are balanced by the block
// scheduler), and the plan's budget of blocks per (layer, kv head).  A
// planned call without a caller's count may use one whole wave of resident
// blocks, shared by its (layer, kv head) pairs, even where that is not a
// multiple of the batch: the grid then grows by up to one block per unit, and
// blocks past the last chunk exit at once.
void set_chunking(const kvq_config* c, int num_splits, int n_layers, int* splits, DecodeArgs* a) {
  const bool rotated = (c->flags & (KVQ_ROTATE_K | KVQ_ROTATE_V)) != 0;
  const int64_t blocks = (int64_t)n_layers * c->batch * c->H_kv * *splits;
  const int64_t resident = (int64_t)sm_count() * (c->D == 128 ? 4 : 2);
  a->fixed_splits = num_splits ? 1 : 0;
  a->min_chunk = num_splits ? 1 : (int)(rotated ? kMinChunkRotated : kMinTilesPerSplit);
  a->chunked = (num_splits || blocks <= 2 * resident) ? 1 : 0;
  a->budget = c->batch * *splits;
  if (a->chunked && !num_splits && *splits > 1) {
    // no more splits per unit than the planning floor allows at full capacity
    const int64_t tiles = (c->max_T + kTile - 1) / kTile + 2;
    const int64_t cap = std::min<int64_t>(std::max<int64_t>(1, tiles / a->min_chunk), kMaxSplits);
    const int64_t wave = resident / ((int64_t)n_layers * c->H_kv);
    const int s2 = (int)std::min<int64_t>((wave + c->batch - 1) / c->batch, cap);
    if (s2 > *splits) {
      a->budget = (int)std::min<int64_t>(wave, (int64_t)c->batch * s2);
      *splits = s2;
    }
  }
}

size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

WsLayout ws_layout(const kvq_config* c) {
  WsLayout w{};
  int g = c->H_q / c->H_kv;
  w.status = 0;
  w.tickets = kWsAlign;
  w.max_units = c->L * c->batch * c->H_kv;
  size_t off = align_up(w.tickets + sizeof(uint32_t) * kTicketsPerUnit * (size_t)w.max_units);
  w.rope = off;
  if (c->flags & KVQ_K_PRE_ROPE) {
    w.rope_base_rows = (c->max_T + kTile - 1) / kTile + 1;
    off = align_up(off + sizeof(float2) * (size_t)(w.rope_base_rows + kRopeExtraRows) * (c->D / 2));
  }
  w.partials = off;
  int64_t mp = 0;
  for (int n = 1; n <= c->L; ++n) {
    int s = splits_for(c, n);
    if (s > 1) {
      int64_t p = (int64_t)n * c->batch * c->H_kv * s;
      if (p > mp) mp = p;
    }
  }
  // explicit split counts up to 64 for one layer are also allowed
  int64_t one = (int64_t)c->batch * c->H_kv * 64;
  if (one > mp) mp = one;
  w.max_partials = (int)mp;
  off = align_up(off + sizeof(float) * (size_t)mp * g * part_row(c->D));
  w.total = off;
  return w;
}

kvq_status check_ws(const kvq_config* c, void* ws, size_t bytes, WsLayout* out) {
  if (!ws) return fail(KVQ_ERR_WORKSPACE, "workspace is NULL");
  WsLayout w = ws_layout(c);
  if (bytes < w.total) return fail(KVQ_ERR_WORKSPACE, "workspace %zu B < %zu B needed", bytes, w.total);
  if (((uintptr_t)ws) % kWsAlign) return fail(KVQ_ERR_WORKSPACE, "workspace not 256-byte aligned");
  *out = w;
  return KVQ_OK;
}

kvq_status cache_ptrs(const kvq_config* c, const kvq_cache* cache, CachePtrs* cp) {
  if (!cache) return fail(KVQ_ERR_ARG, "cache is NULL");
  cp->k_main = (uint8_t*)cache->k_main;
  cp->v_main = (uint8_t*)cache->v_main;
  cp->k_cold = (uint8_t*)cache->k_cold;
  cp->v_cold = (uint8_t*)cache->v_cold;
  cp->k_resid = (uint16_t*)cache->k_resid;
  cp->v_resid = (uint16_t*)cache->v_resid;
  cp->block_table = cache->block_table;
  if (!cp->k_main || !cp->v_main) return fail(KVQ_ERR_ARG, "k_main / v_main is NULL");
  if (c->hot_window > 0 && (!cp->k_cold || !cp->v_cold)) return fail(KVQ_ERR_ARG, "cold buffers are NULL");
  int gam = (c->k_fmt.axis == KVQ_AXIS_CHANNEL || c->v_fmt.axis == KVQ_AXIS_CHANNEL) ? 32 : 1;
  bool ring = !(c->residual_window == 0 && gam == 1);
  if (ring && (!cp->k_resid || !cp->v_resid)) return fail(KVQ_ERR_ARG, "window buffers are NULL");
  if (c->page_tokens > 0 && !cp->block_table) return fail(KVQ_ERR_ARG, "block_table is NULL");
  const uintptr_t any = (uintptr_t)cp->k_main | (uintptr_t)cp->v_main | (uintptr_t)cp->k_cold |
                        (uintptr_t)cp->v_cold | (uintptr_t)cp->k_resid | (uintptr_t)cp->v_resid;
  if (any & 15u) return fail(KVQ_ERR_ARG, "cache buffers must be 16-byte aligned");
  return KVQ_OK;
}

}  // namespace

namespace kvq {

void tbq4_tables(float* centroids, float* thresholds) {
  static float c32[16], t32[15];
  static std::once_flag once;
  std::call_once(once, [] {
    double c[16];
    lloyd_max_normal16(c);
    // the lookup table holds each centroid rounded to fp16 (11 significant
    // bits, nearest, ties to even: every centroid is in fp16's normal range);
    // the thresholds are the exact midpoints of neighbouring entries
    double c16[16];
    for (int i = 0; i < 16; ++i) {
      int e = 0;
      const double m = std::frexp(c[i], &e);  // c = m 2^e, 0.5 <= |m| < 1
      c16[i] = std::ldexp(std::nearbyint(std::ldexp(m, 11)), e - 11);
      c32[i] = (float)c16[i];
    }
    for (int i = 0; i < 15; ++i) t32[i] = (float)(0.5 * (c16[i] + c16[i + 1]));
  });
  std::memcpy(centroids, c32, sizeof(c32));
  std::memcpy(thresholds, t32, sizeof(t32));
}

// The append kernels look TBQ4 indices up in bins holding one midpoint each
// (tbq4_bins.cuh): true when the table's midpoints allow that.
bool tbq4_bins_ok() {
  float c[16], t[15];
  tbq4_tables(c, t);
  const int k0 = tbq4_bin_k0(t);
  for (int e = 0; e < 2 * kTbqBins; ++e) {
    float th;
    int base;
    if (tbq4_bin_entry(t, k0, e, &th, &base) > 1) return false;
  }
  return true;
}

}  // namespace kvq

extern "C" {

const char* kvq_version(void) { return "kvq 0.1 (sm_103a)"; }

const char* kvq_last_error(void) { return g_last_error.c_str(); }

kvq_status kvq_validate_config(const kvq_config* cfg) {
  kvq_status st = check_config(cfg, false);
  return st == KVQ_OK ? ok() : st;
}

kvq_status kvq_block_bytes(int32_t bits, int32_t group, int32_t* bytes) {
  if (!bytes) return fail(KVQ_ERR_ARG, "bytes is NULL");
  if (!valid_bits(bits, true) || (group != 32 && group != 128)) return fail(KVQ_ERR_ARG, "bits=%d group=%d", bits, group);
  *bytes = block_bytes_of(bits, group);
  return ok();
}

kvq_status kvq_bytes_per_token(const kvq_config* cfg, int64_t* bytes) {
  kvq_status st = check_config(cfg, true);
  if (st != KVQ_OK) return st;
  if (!bytes) return fail(KVQ_ERR_ARG, "bytes is NULL");
  const kvq_fmt& kf = cfg->hot_window > 0 ? cfg->k_cold : cfg->k_fmt;
  const kvq_fmt& vf = cfg->hot_window > 0 ? cfg->v_cold : cfg->v_fmt;
  int64_t per_head = 0;
  for (const kvq_fmt* f : {&kf, &vf}) {
    const bool zp = (cfg->flags & (f == &kf ? KVQ_ZP_K : KVQ_ZP_V)) != 0;
    int64_t bb = block_bytes_of(f->bits, f->group) + (zp ? 2 : 0);
    if (f->axis == KVQ_AXIS_TOKEN) {
      per_head += (cfg->D / f->group) * bb;
    } else {
      if ((cfg->D * bb) % f->group) return fail(KVQ_ERR_ARG, "fractional bytes per token");
      per_head += cfg->D * bb / f->group;
    }
  }
  *bytes = (int64_t)cfg->L * cfg->H_kv * per_head;
  return ok();
}

kvq_status kvq_cache_bytes(const kvq_config* cfg, int64_t T, int64_t* bytes) {
  kvq_status st = check_config(cfg, true);
  if (st != KVQ_OK) return st;
  if (!bytes || T < 0) return fail(KVQ_ERR_ARG, "bytes is NULL or T < 0");
  Layout lo = make_layout(cfg);
  int64_t qe = T <= lo.R ? 0 : ((T - lo.R) / lo.gam) * lo.gam;
  int64_t ce = 0;
  if (lo.W > 0 && qe > lo.W) ce = ((qe - lo.W) / lo.gam) * lo.gam;
  int64_t per_head = 0;
  const bool zk = (cfg->flags & KVQ_ZP_K) != 0, zv = (cfg->flags & KVQ_ZP_V) != 0;
  if (lo.W > 0) per_head += fmt_bytes(cfg->k_cold, ce, cfg->D, zk) + fmt_bytes(cfg->v_cold, ce, cfg->D, zv);
  per_head += fmt_bytes(cfg->k_fmt, qe - ce, cfg->D, zk) + fmt_bytes(cfg->v_fmt, qe - ce, cfg->D, zv);
  per_head += 2 * (T - qe) * cfg->D * 2;
  *bytes = (int64_t)cfg->L * cfg->H_kv * per_head;
  return ok();
}

kvq_status kvq_buffer_sizes(const kvq_config* cfg, size_t sizes[6]) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!sizes) return fail(KVQ_ERR_ARG, "sizes is NULL");
  Layout lo = make_layout(cfg);
  size_t per_lbh = (size_t)lo.L * lo.B * lo.H;
  for (int i = 0; i < 6; ++i) sizes[i] = 0;
  if (lo.paged) {
    size_t per_page = (size_t)lo.L * lo.n_pages * lo.H * lo.pt;
    sizes[0] = per_page * lo.kf.row;
    sizes[1] = per_page * lo.vf.row;
  } else {
    sizes[0] = per_lbh * (size_t)lo.rows_k_main * lo.kf.row;
    sizes[1] = per_lbh * (size_t)lo.rows_v_main * lo.vf.row;
  }
  if (lo.tiered) {
    sizes[2] = per_lbh * (size_t)lo.rows_k_cold * lo.kc.row;
    sizes[3] = per_lbh * (size_t)lo.rows_v_cold * lo.vc.row;
  }
  if (lo.ring) {
    sizes[4] = per_lbh * (size_t)lo.ring * lo.D * 2;
    sizes[5] = sizes[4];
  }
  return ok();
}

kvq_status kvq_workspace_bytes(const kvq_config* cfg, size_t* bytes) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!bytes) return fail(KVQ_ERR_ARG, "bytes is NULL");
  *bytes = ws_layout(cfg).total;
  return ok();
}

kvq_status kvq_decode_splits(const kvq_config* cfg, int32_t n_layers, int32_t* splits) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!splits || n_layers < 1 || n_layers > cfg->L) return fail(KVQ_ERR_ARG, "bad n_layers or NULL");
  *splits = splits_for(cfg, n_layers);
  return ok();
}

kvq_status kvq_workspace_init(const kvq_config* cfg, void* workspace, size_t ws_bytes, void* stream) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  WsLayout w;
  if ((st = check_ws(cfg, workspace, ws_bytes, &w)) != KVQ_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(workspace, 0, w.rope, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  if (cfg->flags & KVQ_K_PRE_ROPE) {
    e = launch_rope_tables((float2*)((char*)workspace + w.rope), w.rope_base_rows, cfg->D, cfg->rope_theta, s);
    if (e != cudaSuccess) return cuda_fail(e, "rope table kernel");
  }
  return ok();
}

kvq_status kvq_append(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0, int32_t n_layers,
                      const void* k, const void* v, const int32_t* cu_new, const int32_t* seq_lens,
                      int32_t total_new, int32_t max_new, void* workspace, size_t ws_bytes, void* stream) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > cfg->L)
    return fail(KVQ_ERR_ARG, "layers [%d, %d) outside [0, %d)", layer0, layer0 + n_layers, cfg->L);
  if (total_new < 0 || max_new < 0 || max_new > total_new) return fail(KVQ_ERR_ARG, "total_new / max_new");
  if (max_new > cfg->max_T) return fail(KVQ_ERR_CAPACITY, "max_new=%d > max_T=%d", max_new, cfg->max_T);
  if (total_new > 0 && (!k || !v)) return fail(KVQ_ERR_ARG, "k / v is NULL");
  if (((uintptr_t)k | (uintptr_t)v) & 15u) return fail(KVQ_ERR_ARG, "k / v must be 16-byte aligned");
  if (!cu_new || !seq_lens) return fail(KVQ_ERR_ARG, "cu_new / seq_lens is NULL");
  AppendArgs a{};
  if ((st = cache_ptrs(cfg, cache, &a.cp)) != KVQ_OK) return st;
  WsLayout w;
  if ((st = check_ws(cfg, workspace, ws_bytes, &w)) != KVQ_OK) return st;
  a.lo = make_layout(cfg);
  a.layer0 = layer0;
  a.n_layers = n_layers;
  a.k = (const uint16_t*)k;
  a.v = (const uint16_t*)v;
  a.cu_new = cu_new;
  a.seq_lens = seq_lens;
  a.total_new = total_new;
  a.max_new = max_new;
  a.status = (uint32_t*)((char*)workspace + w.status);
  a.cp.status = a.status;
  cudaError_t e = launch_append(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "append kernels");
  return ok();
}

kvq_status kvq_tbq4_codebook(float centroids[16], float thresholds[15]) {
  if (!centroids || !thresholds) return fail(KVQ_ERR_ARG, "output pointer is NULL");
  tbq4_tables(centroids, thresholds);
  return ok();
}

kvq_status kvq_launch_counts(const kvq_config* cfg, int32_t* append_launches, int32_t* decode_launches) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!append_launches || !decode_launches) return fail(KVQ_ERR_ARG, "output pointer is NULL");
  AppendArgs a{};
  a.lo = make_layout(cfg);
  *append_launches = (a.lo.tiered ? 1 : 0) + (fast_quantize_available(a) ? 2 : 1) + (a.lo.ring ? 1 : 0);
  *decode_launches = 1;
  return ok();
}

kvq_status kvq_commit_lengths(const kvq_config* cfg, const int32_t* cu_new, int32_t* seq_lens, void* stream) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!cu_new || !seq_lens) return fail(KVQ_ERR_ARG, "cu_new / seq_lens is NULL");
  cudaError_t e = launch_commit_lengths(cu_new, seq_lens, cfg->batch, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "commit kernel");
  return ok();
}

// Failure-detection test mode of the tensor-core decode (kvq_test_force_stall).
std::atomic<int> g_stall_polls{0};

// Checks the decode arguments and fills *a (everything but the step).
static kvq_status prep_decode(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0, int32_t n_layers,
                       const void* q, const int32_t* seq_lens, float* out, int32_t num_splits, void* workspace,
                       size_t ws_bytes, DecodeArgs* a) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > cfg->L)
    return fail(KVQ_ERR_ARG, "layers [%d, %d) outside [0, %d)", layer0, layer0 + n_layers, cfg->L);
  if (!q || !seq_lens || !out) return fail(KVQ_ERR_ARG, "q / seq_lens / out is NULL");
  if (num_splits < 0 || num_splits > kMaxSplits) return fail(KVQ_ERR_ARG, "num_splits=%d", num_splits);
  if ((st = cache_ptrs(cfg, cache, &a->cp)) != KVQ_OK) return st;
  WsLayout w;
  if ((st = check_ws(cfg, workspace, ws_bytes, &w)) != KVQ_OK) return st;
  int splits = num_splits ? num_splits : splits_for(cfg, n_layers);
  int64_t units = (int64_t)n_layers * cfg->batch * cfg->H_kv;
  if (splits > 1 && units * splits > w.max_partials)
    return fail(KVQ_ERR_WORKSPACE, "%d splits x %lld units exceed the workspace", splits, (long long)units);
  DecodeArgs planned = *a;
  int grown = splits;
  set_chunking(cfg, num_splits, n_layers, &grown, &planned);
  if (units * grown > w.max_partials) {  // no room for the wider grid: keep the plain budget
    planned.budget = cfg->batch * splits;
    grown = splits;
  }
  splits = grown;
  *a = planned;
  a->lo = make_layout(cfg);
  a->layer0 = layer0;
  a->n_layers = n_layers;
  a->q = (const uint16_t*)q;
  a->seq_lens = seq_lens;
  a->out = out;
  a->splits = splits;
  a->status = (uint32_t*)((char*)workspace + w.status);
  a->cp.status = a->status;
  a->tickets = (uint32_t*)((char*)workspace + w.tickets);
  a->partials = (float*)((char*)workspace + w.partials);
  a->rope = (const float2*)((char*)workspace + w.rope);
  a->rope_base_rows = w.rope_base_rows;
  a->stall_polls = g_stall_polls.load();
  return KVQ_OK;
}

kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0,
                                int32_t n_layers, const void* q, const int32_t* seq_lens, float* out,
                                int32_t num_splits, void* workspace, size_t ws_bytes, void* stream) {
  DecodeArgs a{};
  kvq_status st = prep_decode(cfg, cache, layer0, n_layers, q, seq_lens, out, num_splits, workspace, ws_bytes, &a);
  if (st != KVQ_OK) return st;
  cudaError_t e = launch_decode(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
  return ok();
}

kvq_status kvq_decode_step(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0, int32_t n_layers,
                           const void* k_new, const void* v_new, const void* q, const int32_t* seq_lens,
                           float* out, int32_t num_splits, void* workspace, size_t ws_bytes, void* stream) {
  DecodeArgs a{};
  kvq_status st = prep_decode(cfg, cache, layer0, n_layers, q, seq_lens, out, num_splits, workspace, ws_bytes, &a);
  if (st != KVQ_OK) return st;
  if (!k_new || !v_new) return fail(KVQ_ERR_ARG, "k_new / v_new is NULL");
  if (((uintptr_t)k_new | (uintptr_t)v_new) & 15u) return fail(KVQ_ERR_ARG, "k_new / v_new must be 16-byte aligned");
  AppendArgs& s = a.step;
  s.lo = a.lo;
  s.cp = a.cp;
  s.layer0 = layer0;
  s.n_layers = n_layers;
  s.k = (const uint16_t*)k_new;
  s.v = (const uint16_t*)v_new;
  s.cu_new = nullptr;
  s.seq_lens = seq_lens;
  s.total_new = cfg->batch;
  s.max_new = 1;
  s.status = a.status;
  s.one_per_seq = 1;
  a.len_add = 1;
  cudaError_t e = cudaSuccess;
  if (!launch_decode_step_fused(a, (cudaStream_t)stream, false, &e)) {
    // formats of the generic decode: append, then decode over the new length
    e = launch_append(s, (cudaStream_t)stream);
    if (e == cudaSuccess) e = launch_decode(a, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode step kernels");
  return ok();
}

kvq_status kvq_step_launches(const kvq_config* cfg, int32_t* launches) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (!launches) return fail(KVQ_ERR_ARG, "output pointer is NULL");
  DecodeArgs a{};
  a.lo = make_layout(cfg);
  a.step.lo = a.lo;
  cudaError_t e = cudaSuccess;
  if (launch_decode_step_fused(a, nullptr, true, &e)) {
    *launches = 1;
  } else {
    int32_t app = 0, dec = 0;
    kvq_launch_counts(cfg, &app, &dec);
    *launches = app + dec;
  }
  return ok();
}

kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_cache* cache, int32_t layer, int32_t seq,
                          int32_t t0, int32_t t1, const int32_t* seq_lens, float* k_out, float* v_out,
                          void* workspace, size_t ws_bytes, void* stream) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (layer < 0 || layer >= cfg->L || seq < 0 || seq >= cfg->batch) return fail(KVQ_ERR_ARG, "layer / seq out of range");
  if (t0 < 0 || t1 < t0 || t1 > cfg->max_T) return fail(KVQ_ERR_ARG, "token range [%d, %d)", t0, t1);
  if (!seq_lens || !k_out || !v_out) return fail(KVQ_ERR_ARG, "seq_lens / k_out / v_out is NULL");
  DequantArgs a{};
  if ((st = cache_ptrs(cfg, cache, &a.cp)) != KVQ_OK) return st;
  WsLayout w;
  if ((st = check_ws(cfg, workspace, ws_bytes, &w)) != KVQ_OK) return st;
  if (t1 == t0) return ok();
  a.lo = make_layout(cfg);
  a.layer = layer;
  a.seq = seq;
  a.t0 = t0;
  a.t1 = t1;
  a.seq_lens = seq_lens;
  a.k_out = k_out;
  a.v_out = v_out;
  a.status = (uint32_t*)((char*)workspace + w.status);
  a.cp.status = a.status;
  cudaError_t e = launch_dequantize(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel");
  return ok();
}

kvq_status kvq_test_shrink_bounds(int32_t rows) {
#ifdef KVQ_BOUNDS_CHECK
  if (rows < 0 || rows > (1 << 20)) return fail(KVQ_ERR_ARG, "rows=%d not in [0, 2^20]", rows);
  g_bounds_shrink.store(rows);
  return ok();
#else
  if (rows == 0) return ok();
  return fail(KVQ_ERR_UNSUPPORTED, "bounds checks are compiled into libkvq_checked.so only");
#endif
}

kvq_status kvq_test_force_stall(int32_t polls) {
  if (polls < 0 || polls > (1 << 20)) return fail(KVQ_ERR_ARG, "polls=%d not in [0, 2^20]", polls);
  g_stall_polls.store(polls);
  return ok();
}

kvq_status kvq_read_device_status(const void* workspace, uint32_t* bits, void* stream) {
  if (!workspace || !bits) return fail(KVQ_ERR_ARG, "workspace / bits is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  return ok();
}

kvq_status kvq_clear_device_status(void* workspace, void* stream) {
  if (!workspace) return fail(KVQ_ERR_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kvq_decode_attention_static: decode attention with library-owned scratch,
// for callers that cannot allocate device memory.  The scratch is a fixed
// file-scope device array; its device address is looked up once per device.
// ---------------------------------------------------------------------------

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[KVQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up with
// that device current, once).
kvq_status static_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(KVQ_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_static(const kvq_config* cfg, const kvq_cache* cache, int32_t layer0,
                                                  int32_t n_layers, const void* q, const int32_t* seq_lens,
                                                  float* out, int32_t num_splits, void* stream) {
  kvq_status st = check_config(cfg, false);
  if (st != KVQ_OK) return st;
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > cfg->L)
    return fail(KVQ_ERR_ARG, "layers [%d, %d) outside [0, %d)", layer0, layer0 + n_layers, cfg->L);
  if (!q || !seq_lens || !out) return fail(KVQ_ERR_ARG, "q / seq_lens / out is NULL");
  if (num_splits < 0 || num_splits > kMaxSplits) return fail(KVQ_ERR_ARG, "num_splits=%d", num_splits);
  DecodeArgs a{};
  if ((st = cache_ptrs(cfg, cache, &a.cp)) != KVQ_OK) return st;
  const int plain = num_splits ? num_splits : splits_for(cfg, n_layers);
  int splits = plain;
  set_chunking(cfg, num_splits, n_layers, &splits, &a);
  const int g = cfg->H_q / cfg->H_kv;
  const size_t units = (size_t)n_layers * cfg->batch * cfg->H_kv;
  // this call's scratch: status word, tickets, RoPE tables, split partials
  const size_t off_tickets = kWsAlign;
  size_t off = align_up(off_tickets + sizeof(uint32_t) * kTicketsPerUnit * units);
  const size_t off_rope = off;
  int rope_rows = 0;
  if (cfg->flags & KVQ_K_PRE_ROPE) {
    rope_rows = (cfg->max_T + kTile - 1) / kTile + 1;
    off = align_up(off + sizeof(float2) * (size_t)(rope_rows + kRopeExtraRows) * (cfg->D / 2));
  }
  const size_t off_partials = off;
  auto partials_end = [&](int sp) { return sp > 1 ? align_up(off + sizeof(float) * units * sp * g * part_row(cfg->D)) : off; };
  if (splits != plain && partials_end(splits) > (size_t)KVQ_STATIC_SCRATCH_BYTES) {
    splits = plain;  // no room for the wider grid: keep the plain budget
    a.budget = cfg->batch * plain;
  }
  off = partials_end(splits);
  if (off > (size_t)KVQ_STATIC_SCRATCH_BYTES)
    return fail(KVQ_ERR_WORKSPACE, "this call needs %zu B of scratch; the static scratch holds %u B", off,
                (unsigned)KVQ_STATIC_SCRATCH_BYTES);
  void* base = nullptr;
  if ((st = static_scratch(&base)) != KVQ_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // status word and tickets must start at zero; the rest is overwritten
  cudaError_t e = cudaMemsetAsync(base, 0, off_rope, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  if (rope_rows) {
    e = launch_rope_tables((float2*)((char*)base + off_rope), rope_rows, cfg->D, cfg->rope_theta, s);
    if (e != cudaSuccess) return cuda_fail(e, "rope table kernel");
  }
  a.lo = make_layout(cfg);
  a.layer0 = layer0;
  a.n_layers = n_layers;
  a.q = (const uint16_t*)q;
  a.seq_lens = seq_lens;
  a.out = out;
  a.splits = splits;
  a.status = (uint32_t*)base;
  a.cp.status = a.status;
  a.tickets = (uint32_t*)((char*)base + off_tickets);
  a.partials = (float*)((char*)base + off_partials);
  a.rope = (const float2*)((char*)base + off_rope);
  a.rope_base_rows = rope_rows;
  a.stall_polls = g_stall_polls.load();
  e = launch_decode(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
  return ok();
}
