// Split-K decode attention on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulators):
//   K per-channel 4/2-bit over 32-token groups, or per-token 8/4/3-bit blocks;
//   V per-token 8/4/3/2-bit blocks; an optional fp16 window; a hot/cold pair
//   of per-channel formats; keys stored pre-RoPE (split-half RoPE applied in
//   the kernel); optional rotation (no window then); contiguous or 16/32-token
//   pages.
//
// Per 32-token group the scores are S^T[token][col] = K[token][d] Q^T[d][col]
// with tokens on M and, on N, the query heads sharing the kv head, each head
// twice: column 2h holds the fp16 part ("hi") of head h's query and column
// 2h+1 the fp16 remainder ("lo"), so q = hi + lo to about 22 bits.  The PV
// product is O^T[d][col] = V^T[d][token] P^T[token][col] with the same hi/lo
// split of the probabilities.  Codes enter the tensor cores as exact fp16
// integers; block scales multiply the fp32 scores (per-token K), the query
// (per-channel K) or the probabilities (per-token V).  This is the rotated-
// domain attention of trefon.com "Matematyka cache KV" ("najpierw obrot":
// rotate the query once, read blocks as code x scale, rotate the output back
// once) with nalar.dev's s_i = q.k_i / sqrt(D) and output = sum_i p_i v_i.
//
// Pre-RoPE keys (troisinh.com "KV Cache Quantization", "RoPE - Cai bay tinh
// vi"; split-half pairs as lehuy.net "NexusQuant" lists): with t = t0 + j in a
// group starting at t0, q . R(t) k = (R(-t0) q) . (R(j) k).  The query is
// turned by -t0 once per group; each key value is dequantized, turned by its
// in-group offset j and split into fp16 hi + lo, so the product keeps ~22
// bits on both sides.  Angles come from fp64 tables in the workspace.
//
// Layout of one group: M-tile mu (0, 1) row r is token
// tau(mu, r) = 4(r & 7) + 2mu + (r >> 3); k-chunk kc = 2s + b (span s of 32
// channels) pairs channels (c, c+4) in k-slots (2t, 2t+1) and (c+1, c+5) in
// (2t+8, 2t+9), c = 32s + 8t + 2b (t = lane % 4), so channel c + D/2 sits in
// k-chunk kc + D/32 at the same slot (the RoPE partner); d-tile (s, e) row r
// is channel 32s + 4(r & 7) + 2e + (r >> 3).
//
// Work split: CTA = 4 warps on one chunk of tiles of one (layer, sequence,
// kv head) (see plan_work); each warp streams its own groups through a ring of 2 or 3 shared-memory
// stages filled by 1-D bulk copies (TMA engine) that complete on per-stage
// mbarriers, and keeps its own online softmax; warps merge in shared memory and splits merge in
// the workspace (the last CTA to take a ticket combines; nobody waits).
#pragma once

#include "append_generic.cuh"
#include "split_combine.cuh"

namespace kvq {

cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s);

namespace {

// KF_TQ / VF_TQ: TBQ4 blocks (4-bit indices into the 16-entry fp16 table).
enum : int { KF_CH4 = 0, KF_T8 = 1, KF_T4 = 2, KF_T3 = 3, KF_CH2 = 4, KF_TQ = 5 };
enum : int { VF_T8 = 0, VF_T4 = 1, VF_T3 = 2, VF_T2 = 3, VF_TQ = 4 };

constexpr int kWarps = 4;
constexpr int kThreadsMma = kWarps * 32;
constexpr int kMaxStages = 3;  // per-warp bulk-copy ring depth (Cfg::STAGES), at most
constexpr float kLog2eF = 1.4426950408889634f;

constexpr int bits_k(int kf) { return kf == KF_T8 ? 8 : kf == KF_T3 ? 3 : kf == KF_CH2 ? 2 : 4; }
constexpr int bits_v(int vf) { return vf == VF_T8 ? 8 : vf == VF_T3 ? 3 : vf == VF_T2 ? 2 : 4; }
constexpr int align16(int x) { return (x + 15) / 16 * 16; }
__host__ __device__ constexpr float code_bias(int bits) { return (float)(1 << (bits - 1)); }  // symmetric storage bias

// Byte geometry of one tier's formats.  Z: asymmetric blocks (fp16 scale,
// fp16 zero, codes 0..2^b-1) for K and V.  The code unpackers return the
// field minus the symmetric storage bias beta = 2^(b-1), so an asymmetric
// value c s + z is read as (c - beta) s + (z + beta s): the codes take the
// symmetric path unchanged and the zero z' = z + beta s adds a term per block.
template <int D, int KF_, int KG_, int VF_, int VG_, bool Z_ = false>
struct Tier {
  static constexpr int KF = KF_, KG = KG_, VF = VF_, VG = VG_;
  static constexpr bool Z = Z_;
  static constexpr int KB = bits_k(KF), VB = bits_v(VF);
  static constexpr bool KCH = KF == KF_CH4 || KF == KF_CH2;
  static constexpr bool KLUT = KF == KF_TQ, VLUT = VF == VF_TQ;  // codes index the TBQ4 table
  static constexpr int HDR = Z ? 4 : 2;                     // block header bytes
  static constexpr int KBB = HDR + (KCH ? 32 : KG) * KB / 8;  // block bytes
  static constexpr int VBB = HDR + VG * VB / 8;
  static constexpr int KROW = KCH ? D * KBB : (D / KG) * KBB;  // group row / token row
  static constexpr int VROW = (D / VG) * VBB;
  static constexpr int KSTAGE = KCH ? KROW : 32 * KROW;
  static constexpr int VSTAGE = 32 * VROW;
  static constexpr int KSPB = KCH ? 1 : KG / 32;  // spans per K block
  static constexpr int VSPB = VG / 32;
  static constexpr int KSPAN = 32 * KB / 8;  // code bytes of a span of one token
  static constexpr int VSPAN = 32 * VB / 8;
  static_assert(!Z || (KCH && VG == 32 && !KLUT && !VLUT), "asymmetric blocks: per-channel K, 32-value V blocks");
};

constexpr int cmax(int a, int b) { return a > b ? a : b; }

// HOT: the only tier (COLD_ = false) or the hot tier; COLD: the cold tier.
// HC: the MMA columns are the query heads themselves (8 per n-tile) and the
// query / probability hi and lo parts are two B fragments accumulated into the
// same C (for groups of more than 4 heads: the same MMAs as hi / lo columns,
// half the accumulators).  Otherwise column 2h is head h's hi part and 2h + 1
// its lo part.
template <int D_, int NT_, class HOT_, class COLD_, bool HAS_COLD_, bool ROPE_, bool HC_ = false>
struct Cfg {
  static constexpr int D = D_, NT = NT_;
  static constexpr bool HC = HC_;
  static constexpr int J = HC ? 2 : 1;  // heads per lane per n-tile
  using HOT = HOT_;
  using COLD = COLD_;
  static constexpr bool HAS_COLD = HAS_COLD_, ROPE = ROPE_;
  static constexpr bool Z = HOT::Z;
  static_assert(!HAS_COLD || COLD::Z == HOT::Z, "both tiers asymmetric or neither");
  static_assert(!HC || (!HOT::KCH && !ROPE && !Z && !HAS_COLD && NT == 1), "heads as columns: per-token K only");
  static constexpr int KSTAGE = HAS_COLD ? cmax(HOT::KSTAGE, COLD::KSTAGE) : HOT::KSTAGE;
  static constexpr int VSTAGE = HAS_COLD ? cmax(HOT::VSTAGE, COLD::VSTAGE) : HOT::VSTAGE;
  static constexpr int VOFF = align16(KSTAGE + 16);
  static constexpr int STAGE = VOFF + align16(VSTAGE + 16);
  static constexpr int KC = D / 16;  // k-chunks
  static constexpr int NS = D / 32;  // spans
  // per-lane query fragments (+ fp32 query for RoPE, + fp32 query by head for
  // the zero terms, + the lo fragments with heads as columns)
  static constexpr bool QH = HOT::KCH || (HAS_COLD && COLD::KCH);  // query half pairs (per-channel K)
  // per-token K codes read as fp16 subnormals (see k_token_pairs): one tier of
  // 8-, 4- or 3-bit uniform codes; KBLK K blocks per token row
  static constexpr bool KSUB = !HOT::KCH && !HOT::KLUT && !HAS_COLD && !ROPE && !Z &&
                               (HOT::KB == 8 || HOT::KB == 4 || HOT::KB == 3);
  static constexpr int KBLK = HOT::KCH ? 1 : D / HOT::KG;
  // V codes read as subnormals (see v_pair4): one tier of 8-, 4- or 2-bit
  // uniform codes, symmetric or asymmetric (the bias MMA leaves field - beta;
  // the zero term adds z' = z + beta s), not with heads as columns (there the
  // bias MMAs of the hi and lo fragments cost more than the conversions they
  // replace); NBV V blocks per token row
  static constexpr bool VSUB =
      !HAS_COLD && !HC && !HOT::VLUT && (HOT::VB == 8 || HOT::VB == 4 || HOT::VB == 2);
  static constexpr int NBV = D / HOT::VG;
  static constexpr int QSM = KC * NT * 32 * (8 + (QH ? 8 : 0) + (ROPE ? 16 : 0) + (Z ? 8 : 0) + (HC ? 8 : 0)) +
                             (KSUB ? 4 * KBLK * NT * 8 : 0);
  static constexpr int MIN_CTAS = D == 128 ? 4 : 2;  // CTAs per SM the register budget aims at
  // groups in flight per warp: one consumed while STAGES - 1 land (D = 256 runs two CTAs per SM,
  // so each warp keeps two groups in flight)
  static constexpr int STAGES = D == 256 ? 3 : 2;
  static_assert(STAGES <= kMaxStages, "stage count");
  static constexpr int SMEM = QSM + kWarps * STAGES * STAGE;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// fp16 pair (lo half = a, hi half = b), round to nearest.
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float rn16(float x) { return __half2float(__float2half_rn(x)); }

// fp16 part of x (hi) or the remainder x - hi (lo), as fp32.
__device__ __forceinline__ float split_part(float x, bool lo) {
  const float hi = rn16(x);
  return lo ? x - hi : hi;
}

// ---- bulk copies (TMA engine) completing on a per-stage mbarrier ----------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes the barrier initialization visible to the async proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Orders this thread's earlier shared-memory accesses (generic proxy) before
// later bulk copies into the same bytes (async proxy).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// `bytes` (a multiple of 16) from global `src` to shared `dst`, both 16-byte
// aligned; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`; false when the limit ran out
// (the same answer on every lane of the warp).
constexpr int kSpinLimit = 1 << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit = kSpinLimit) {
  bool ok = false;
  for (int i = 0; i < limit && !ok; ++i) ok = mbar_test(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }
// four bytes at an even address
__device__ __forceinline__ uint32_t ld_u32e(const uint8_t* p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }
// 32 bits of a row's bit stream from bit 8 off + lb on, where the row is
// 4-byte aligned, off a byte offset that is a constant after unrolling and lb
// the lane's bit offset: two aligned words funnel-shifted (the word after the
// field lies inside the stage buffer).  The word index and shift depend on
// off mod 4 and the lane only, so they are computed once per lane.
__device__ __forceinline__ uint32_t ld_bits(const uint8_t* row, int off, int lb) {
  const int t = 8 * (off & 3) + lb;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(row + (off & ~3)) + (t >> 5);
  return __funnelshift_r(w[0], w[1], (uint32_t)t);
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// fp16 bits of -n for an integer 1 <= n < 2048 (exact).
__host__ __device__ constexpr uint32_t neg_f16_bits(int n) {
  int e = 0;
  while ((2 << e) <= n) ++e;  // 2^e <= n < 2^(e+1)
  return 0x8000u | (uint32_t)(e + 15) << 10 | (uint32_t)((n - (1 << e)) << (10 - e));
}

// Two codes of B bits at bit B*j of each 16-bit half of x, as an exact fp16
// pair (code with the storage bias beta = 2^(B-1) removed).  A field inside
// the fp16 mantissa (bits 0..9) is masked in place: 1024 + c 2^(Bj), times
// 2^-(Bj), minus 2^(10 - Bj) + beta, is c - beta exactly (one fma); a field
// reaching bit 10 is shifted down first.
template <int B>
__device__ __forceinline__ uint32_t code_pair(uint32_t x, int j) {
  constexpr uint32_t m = (1u << B) - 1, beta = 1u << (B - 1);
  if (j == 0) return hsub2u((x & (m * 0x00010001u)) | 0x64006400u, (0x6400u + beta) * 0x00010001u);
  if (B * j + B <= 10) {
    const int sh = B * j;
    const uint32_t scale = (uint32_t)(15 - sh) << 10;  // 2^-sh
    const uint32_t off = neg_f16_bits((1 << (10 - sh)) + (int)beta);
    return hfma2u((x & ((m << sh) * 0x00010001u)) | 0x64006400u, scale * 0x00010001u, off * 0x00010001u);
  }
  return hsub2u(((x >> (B * j)) & (m * 0x00010001u)) | 0x64006400u, (0x6400u + beta) * 0x00010001u);
}

// Eight 4-bit codes, four per 16-bit half of x (nibble j of each half), as
// the fp16 pairs r[j] = (low-half code j, high-half code j) - 8.  Nibbles 0
// and 2 go through 1024 + n; nibbles 1 and 3 through 1024 + 16n, scaled by
// 1/16 and offset by -72 in one exact fma.
__device__ __forceinline__ void dq4(uint32_t x, uint32_t (&r)[4]) {
  r[0] = hsub2u((x & 0x000F000Fu) | 0x64006400u, 0x64086408u);
  r[1] = hfma2u((x & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
  x >>= 8;
  r[2] = hsub2u((x & 0x000F000Fu) | 0x64006400u, 0x64086408u);
  r[3] = hfma2u((x & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
}

// Two int8 codes in byte 0 of each 16-bit half of (x >> 8j).
__device__ __forceinline__ uint32_t code_pair8(uint32_t x, int j) {
  return hsub2u(((x >> (8 * j)) & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}

// Eight TBQ4 indices, four per 16-bit half of x (nibble j of each half), as
// the fp16 pairs r[j] = (T[low-half nibble j], T[high-half nibble j]) of the
// 16-entry table T.  T is symmetric (T[15 - k] = -T[k]), so an index k maps to
// the magnitude M[k ^ (k < 8 ? 7 : 0) & 7] = T[8 + ...] with the sign of
// bit 3; lut holds the low bytes (lut[0], lut[1]) and high bytes (lut[2],
// lut[3]) of the eight magnitudes, looked up four at a time by byte permutes.
__device__ __forceinline__ void dqt(uint32_t x, uint32_t (&r)[4], const uint32_t (&lut)[4]) {
  const uint32_t neg = ~x & 0x88888888u;                         // bit 3 clear: negative entry
  const uint32_t mx = (x ^ ((neg >> 3) * 7u)) & 0x77777777u;     // magnitude index per nibble
  const uint32_t a = mx & 0x0F0F0F0Fu, b = (mx >> 4) & 0x0F0F0F0Fu;
  const uint32_t c = a | (a >> 12), d = b | (b >> 12);           // byte0: (m0, m4), byte1: (m2, m6) | (m1, m5), (m3, m7)
  const uint32_t sel[2] = {__byte_perm(c, d, 0x0040), __byte_perm(c, d, 0x0051)};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t lo = __byte_perm(lut[0], lut[1], sel[h]);     // low bytes of 4 entries
    const uint32_t hi = __byte_perm(lut[2], lut[3], sel[h]);     // high bytes
    const uint32_t p0 = __byte_perm(lo, hi, 0x5140), p1 = __byte_perm(lo, hi, 0x7362);
    const int j0 = 2 * h, j1 = 2 * h + 1;
    r[j0] = p0 | ((neg << (12 - 4 * j0)) & 0x80008000u);
    r[j1] = p1 | ((neg << (12 - 4 * j1)) & 0x80008000u);
  }
}

// Codes read as fp16 subnormals: a 16-bit field p below 0x800 is the fp16
// value p 2^-24 exactly (subnormals and the first binade are one linear
// scale), and the tensor cores multiply subnormal operands exactly.  So a
// biased code n masked in place at bit position sh is the exact operand
// n 2^sh 2^-24, one logic operation per pair and no conversion.  The 2^sh of
// each position is taken out of the query fragment that meets it, the 2^-24
// out of the score, and the storage bias beta by subtracting beta times the
// sum of that query fragment (one constant per K block and column).
// k_sub_shift(bits, odd_chunk, b1): log2 of the factor the codes meeting query
// fragment b1 (else b0) of an odd (else even) k-chunk carry.
__host__ __device__ constexpr int k_sub_shift(int bits, bool odd_chunk, bool b1) {
  return bits == 4 ? (b1 ? 4 : 0) : bits == 3 ? (odd_chunk ? 6 : (b1 ? 3 : 0)) : 0;
}
__host__ __device__ constexpr int k_sub_bias(int bits) { return bits == 8 ? 128 : 1 << (bits - 1); }

// v_sub_shift(bits, j): log2 of the factor the V code of channel 4 gq + j of
// a span carries (4-bit nibbles in place: 0, 4, 0, 4; 2-bit fields 0, 2, 4, 6).
__host__ __device__ constexpr int v_sub_shift(int bits, int j) {
  return bits == 4 ? ((j & 1) ? 4 : 0) : bits == 2 ? 2 * j : 0;
}
// fp16 pair of -beta 2^v_sub_shift 2^-24 (a negative subnormal, exact).
__host__ __device__ constexpr uint32_t v_sub_neg(int bits, int j) {
  return (0x8000u | ((uint32_t)(1 << (bits - 1)) << v_sub_shift(bits, j))) * 0x00010001u;
}

// A query fragment pair (b0, b1) of an even (ODD = false) or odd k-chunk with
// the position factors of the subnormal codes multiplied back in.
template <int BITS, bool ODD>
__device__ __forceinline__ uint2 unsub_frag(uint2 q) {
  constexpr int s0 = k_sub_shift(BITS, ODD, false), s1 = k_sub_shift(BITS, ODD, true);
  constexpr uint32_t h0 = (uint32_t)(15 + s0) << 10, h1 = (uint32_t)(15 + s1) << 10;  // fp16 2^s
  if constexpr (s0 != 0) q.x = hmul2u(q.x, h0 * 0x00010001u);
  if constexpr (s1 != 0) q.y = hmul2u(q.y, h1 * 0x00010001u);
  return q;
}

// Eight 3-bit K codes (channels c0..c0+7 of one token, bits 24 tq of the span
// at byte off of the 4-byte aligned row) as four fp16 pairs (c0+j, c0+j+4);
// SUB: biased codes as subnormals at bit positions 0, 3, 6, 6.
template <bool SUB = false>
__device__ __forceinline__ void k_token_pairs3(const uint8_t* row, int off, int tq, uint32_t (&r)[4]) {
  const uint32_t w = ld_bits(row, off, 24 * tq);
  const uint32_t x = (w & 0xFFFu) | ((w << 4) & 0x0FFF0000u);
  if constexpr (SUB) {
    r[0] = x & 0x00070007u;
    r[1] = x & 0x00380038u;
    r[2] = x & 0x01C001C0u;
    r[3] = (x >> 3) & 0x01C001C0u;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = code_pair<3>(x, j);
  }
}

// Eight K codes (channels c0..c0+7 of one token) as four fp16 pairs
// (c0+j, c0+j+4), j = 0..3.  `p` points at the first code byte of the span.
// SUB: biased codes as subnormals (4-bit: nibbles in place, positions 0 and
// 4; 8-bit: the int8 code with its sign bit flipped, position 0).
template <class C, bool SUB = false>
__device__ __forceinline__ void k_token_pairs(const uint8_t* p, int tq, uint32_t (&r)[4], const uint32_t (&lut)[4]) {
  if constexpr (C::KLUT) {
    dqt(ld_u32e(p + 4 * tq), r, lut);
  } else if constexpr (C::KB == 4) {
    const uint32_t x = ld_u32e(p + 4 * tq);
    if constexpr (SUB) {
      r[0] = x & 0x000F000Fu;
      r[1] = x & 0x00F000F0u;
      r[2] = (x >> 8) & 0x000F000Fu;
      r[3] = (x >> 8) & 0x00F000F0u;
    } else {
      dq4(x, r);
    }
  } else if constexpr (C::KB == 8) {
    const uint32_t w0 = ld_u32e(p + 8 * tq), w1 = ld_u32e(p + 8 * tq + 4);
    const uint32_t xa = __byte_perm(w0, w1, 0x5410), xb = __byte_perm(w0, w1, 0x7632);
    if constexpr (SUB) {
      r[0] = (xa & 0x00FF00FFu) ^ 0x00800080u;
      r[1] = ((xa >> 8) & 0x00FF00FFu) ^ 0x00800080u;
      r[2] = (xb & 0x00FF00FFu) ^ 0x00800080u;
      r[3] = ((xb >> 8) & 0x00FF00FFu) ^ 0x00800080u;
    } else {
      r[0] = code_pair8(xa, 0);
      r[1] = code_pair8(xa, 1);
      r[2] = code_pair8(xb, 0);
      r[3] = code_pair8(xb, 1);
    }
  } else {
    static_assert(C::KB != 3, "3-bit K codes: k_token_pairs3");
  }
}

// Four V codes (channels 4*gq..4*gq+3 of a span) of token rows ra and rb as
// four fp16 pairs (row a, row b) for channel 4gq+j.  p* point at the span's
// first code byte of each row.
// SUB: biased codes as subnormals at the positions of v_sub_shift.
template <class C, bool SUB = false>
__device__ __forceinline__ void v_pair4(const uint8_t* pa, const uint8_t* pb, int gq, uint32_t (&r)[4],
                                        const uint32_t (&lut)[4]) {
  if constexpr (C::VB == 8) {
    const uint32_t wa = ld_u32e(pa + 4 * gq), wb = ld_u32e(pb + 4 * gq);
    const uint32_t xa = __byte_perm(wa, wb, 0x5410), xb = __byte_perm(wa, wb, 0x7632);
    if constexpr (SUB) {
      r[0] = (xa & 0x00FF00FFu) ^ 0x00800080u;
      r[1] = ((xa >> 8) & 0x00FF00FFu) ^ 0x00800080u;
      r[2] = (xb & 0x00FF00FFu) ^ 0x00800080u;
      r[3] = ((xb >> 8) & 0x00FF00FFu) ^ 0x00800080u;
    } else {
      r[0] = code_pair8(xa, 0);
      r[1] = code_pair8(xa, 1);
      r[2] = code_pair8(xb, 0);
      r[3] = code_pair8(xb, 1);
    }
  } else {
    static_assert(C::VB != 3, "3-bit V codes: v_pair4_3");
    uint32_t ua, ub;
    if constexpr (C::VB == 4) {
      ua = ld_u16(pa + 2 * gq);
      ub = ld_u16(pb + 2 * gq);
    } else {  // 2 bits: byte gq of the span
      ua = pa[gq];
      ub = pb[gq];
    }
    const uint32_t x = __byte_perm(ua, ub, 0x5410);
    if constexpr (C::VLUT) {
      dqt(x, r, lut);
    } else if constexpr (SUB && C::VB == 4) {
      r[0] = x & 0x000F000Fu;
      r[1] = x & 0x00F000F0u;
      r[2] = (x >> 8) & 0x000F000Fu;
      r[3] = (x >> 8) & 0x00F000F0u;
    } else if constexpr (SUB) {  // 2 bits
      r[0] = x & 0x00030003u;
      r[1] = x & 0x000C000Cu;
      r[2] = x & 0x00300030u;
      r[3] = x & 0x00C000C0u;
    } else if constexpr (C::VB == 4) {
      dq4(x, r);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) r[j] = code_pair<C::VB>(x, j);
    }
  }
}

// Four 3-bit V codes (channels 4 gq .. 4 gq + 3: bits 12 gq of the span at
// byte off) of the 4-byte aligned token rows ra and rb as four fp16 pairs
// (row a, row b).  Bits 12..15 of each half hold the next lane's codes, which
// the field masks of code_pair drop.
__device__ __forceinline__ void v_pair4_3(const uint8_t* ra, const uint8_t* rb, int off, int gq, uint32_t (&r)[4]) {
  const uint32_t x = __byte_perm(ld_bits(ra, off, 12 * gq), ld_bits(rb, off, 12 * gq), 0x5410);
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = code_pair<3>(x, j);
}

template <class C>
struct WarpState {
  float o[C::KC][C::NT][4];
  float m[C::NT * C::J], l[C::NT * C::J];  // per (n-tile, head of the lane)
  // asymmetric V: sum over this lane's tokens of p z' per 32-channel block
  // (for the lane's head 4 nt + tq), rescaled with o
  float zo[C::Z ? C::NS : 1][C::NT];
};

// Subnormal V codes: the output so far from 2^-24 units with position factors
// (row gq of d-tile (s, e) holds channel 4 gq + 2 e, row gq + 8 channel
// 4 gq + 2 e + 1 of span s) back to plain units.  Linear in o, so it may run
// at any point between groups; it runs once per warp, before any 16-bit
// window group adds plain products.
template <class C>
__device__ __forceinline__ void vsub_finish(WarpState<C>& ws) {
  if constexpr (C::VSUB) {
    constexpr int VB = C::HOT::VB;
#pragma unroll
    for (int sp = 0; sp < C::NS; ++sp)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ws.o[2 * sp + e][nt][k] *= ldexpf(1.f, 24 - v_sub_shift(VB, 2 * e + (k >> 1)));
          }
  }
}

// Online softmax over one group's scores; returns the probabilities of the
// thread's four tokens 4gq..4gq+3 for each n-tile.
template <class C>
__device__ __forceinline__ void online_softmax(WarpState<C>& ws, float (&S)[2][C::NT][4], int n_valid, int gq,
                                               float qscale, float (&p)[C::NT][C::J][4]) {
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
    for (int j = 0; j < C::J; ++j) {
      float s[4];
      if constexpr (C::HC) {  // column 2tq + j is head 8 nt + 2 tq + j
        s[0] = S[0][nt][j] * qscale;
        s[1] = S[0][nt][2 + j] * qscale;
        s[2] = S[1][nt][j] * qscale;
        s[3] = S[1][nt][2 + j] * qscale;
      } else {  // columns 2tq (hi) + 2tq + 1 (lo): head 4 nt + tq
        s[0] = (S[0][nt][0] + S[0][nt][1]) * qscale;
        s[1] = (S[0][nt][2] + S[0][nt][3]) * qscale;
        s[2] = (S[1][nt][0] + S[1][nt][1]) * qscale;
        s[3] = (S[1][nt][2] + S[1][nt][3]) * qscale;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (4 * gq + k >= n_valid) s[k] = -INFINITY;
        mx = fmaxf(mx, s[k]);
      }
      const int si = nt * C::J + j;
      if (__all_sync(0xffffffffu, mx <= ws.m[si])) {
        // no score above the running maximum: it stays, so the update is
        // p = 2^(s - m), l += sum p (what the full update below gives when
        // its maximum does not move), without the cross-lane reduction
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          p[nt][j][k] = exp2f(s[k] - ws.m[si]);
          sum += p[nt][j][k];
        }
        ws.l[si] += sum;
        continue;
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(ws.m[si], mx);
      const float alpha = exp2f(ws.m[si] - m_new);
      ws.m[si] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        p[nt][j][k] = exp2f(s[k] - m_new);
        sum += p[nt][j][k];
      }
      ws.l[si] = ws.l[si] * alpha + sum;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int i = 0; i < C::KC; ++i) {
          if constexpr (C::HC) {
            ws.o[i][nt][j] *= alpha;
            ws.o[i][nt][2 + j] *= alpha;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) ws.o[i][nt][e] *= alpha;
          }
        }
        if constexpr (C::Z) {
#pragma unroll
          for (int s2 = 0; s2 < C::NS; ++s2) ws.zo[s2][nt] *= alpha;
        }

      }
    }
  }
}

// P^T fragments of M-tile mu, n-tile nt: probabilities times the per-token
// value scales sa (row gq) / sb (row gq+8), split into fp16 hi/lo columns and
// transposed with movmatrix into the B layout.
__device__ __forceinline__ void p_fragments(float pa, float pb, uint32_t& b0, uint32_t& b1) {
  const float ha = rn16(pa), hb = rn16(pb);
  b0 = movtrans(pack_h2(ha, pa - ha));
  b1 = movtrans(pack_h2(hb, pb - hb));
}

// Heads as columns: the probabilities pA, pB of one token for the lane's two
// heads (columns 2tq, 2tq + 1) as the hi and the lo B fragments.
__device__ __forceinline__ void p_fragments_hc(float pA, float pB, uint32_t& hi, uint32_t& lo) {
  const float hA = rn16(pA), hB = rn16(pB);
  hi = movtrans(pack_h2(hA, hB));
  lo = movtrans(pack_h2(pA - hA, pB - hB));
}

// Per-thread context of the decode kernel shared with its helpers.
template <class C>
struct Ctx {
  int gq, tq, lane, g;
  bool lo_part;
  uint32_t lo_mask;
  const uint2* qb;        // [KC][NT][32]: B fragments (hi or lo part; hi with heads as columns)
  const uint2* qbl;       // [KC][NT][32]: lo B fragments (heads as columns)
  const uint2* qh;        // [KC][NT][32]: query half pairs
  const float4* qr;       // [KC][NT][32]: fp32 query (RoPE)
  const float* qz;        // [4 NT][D]: fp32 query by head, zero past g (asymmetric K)
  const float* kq;        // [KBLK][NT][8 columns]: beta times the column's query sum per K block (KSUB)
  const float2* rope_base;
  const float4* rope_frag;  // [KC/2][4 tokens k][2 pairs][32 lanes]: (cos, cos, sin, sin) of R(j), lane's channels
  const uint4* rope_tab;    // [KC/2][4 tokens k][32 lanes][2]: fp16 hi / lo cos and sin of R(j), lane's channel pairs
  uint32_t lut[4];          // TBQ4 table magnitudes: low bytes (2 words), high bytes (2 words)
};

// B fragments of the query turned by -t0 (pre-RoPE keys) for the k-chunk
// pair (kcp, kcp + KC/2): lower channel c and its partner c + D/2.
template <class C>
__device__ __forceinline__ void rope_query_pair(const Ctx<C>& cx, const float2* base, int kcp,
                                                uint32_t (&ql)[C::NT][2], uint32_t (&qu)[C::NT][2]) {
  constexpr int NT = C::NT, KC = C::KC;
  const int c = 32 * (kcp >> 1) + 8 * cx.tq + 2 * (kcp & 1);
  const float2 f0 = __ldg(base + c), f1 = __ldg(base + c + 4), f2 = __ldg(base + c + 1), f3 = __ldg(base + c + 5);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float4 l = cx.qr[(kcp * NT + nt) * 32 + cx.lane], u = cx.qr[((kcp + KC / 2) * NT + nt) * 32 + cx.lane];
    const float l0 = l.x * f0.x + u.x * f0.y, u0 = u.x * f0.x - l.x * f0.y;
    const float l1 = l.y * f1.x + u.y * f1.y, u1 = u.y * f1.x - l.y * f1.y;
    const float l2 = l.z * f2.x + u.z * f2.y, u2 = u.z * f2.x - l.z * f2.y;
    const float l3 = l.w * f3.x + u.w * f3.y, u3 = u.w * f3.x - l.w * f3.y;
    ql[nt][0] = pack_h2(split_part(l0, cx.lo_part), split_part(l1, cx.lo_part));
    ql[nt][1] = pack_h2(split_part(l2, cx.lo_part), split_part(l3, cx.lo_part));
    qu[nt][0] = pack_h2(split_part(u0, cx.lo_part), split_part(u1, cx.lo_part));
    qu[nt][1] = pack_h2(split_part(u2, cx.lo_part), split_part(u3, cx.lo_part));
  }
}

// The query turned by -t0 (pre-RoPE keys), fp32, for the k-chunk pair (kcp,
// kcp + KC/2): l[nt] = lower channels (c, c + 4, c + 1, c + 5), u[nt] their
// partners c + D/2, ..., for the lane's head of n-tile nt.
template <class C>
__device__ __forceinline__ void rope_query_f32(const Ctx<C>& cx, const float2* base, int kcp, float4 (&l)[C::NT],
                                               float4 (&u)[C::NT]) {
  constexpr int NT = C::NT, KC = C::KC;
  const int c = 32 * (kcp >> 1) + 8 * cx.tq + 2 * (kcp & 1);  // even: (c, c + 1) is one 16-byte load
  const float4 f02 = __ldg(reinterpret_cast<const float4*>(base + c));
  const float4 f13 = __ldg(reinterpret_cast<const float4*>(base + c + 4));
  const float2 f0 = make_float2(f02.x, f02.y), f2 = make_float2(f02.z, f02.w);
  const float2 f1 = make_float2(f13.x, f13.y), f3 = make_float2(f13.z, f13.w);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float4 a = cx.qr[(kcp * NT + nt) * 32 + cx.lane], b = cx.qr[((kcp + KC / 2) * NT + nt) * 32 + cx.lane];
    l[nt] = make_float4(a.x * f0.x + b.x * f0.y, a.y * f1.x + b.y * f1.y, a.z * f2.x + b.z * f2.y,
                        a.w * f3.x + b.w * f3.y);
    u[nt] = make_float4(b.x * f0.x - a.x * f0.y, b.y * f1.x - a.y * f1.y, b.z * f2.x - a.z * f2.y,
                        b.w * f3.x - a.w * f3.y);
  }
}

// fp16 pair of the packed fp32 pair X for this lane's B column: the values
// rounded to fp16 (NM = (-0, -0): hi columns) or the fp16 rounding of their
// remainders x - fp16(x) (NM = (-1, -1): lo columns); x - fp16(x) is exact in
// fp32.
__device__ __forceinline__ uint32_t col_pair(uint64_t X, uint64_t NM) {
  float x0, x1;
  upk2(X, x0, x1);
  const float2 b = __half22float2(__floats2half2_rn(x0, x1));
  float r0, r1;
  upk2(fma2(NM, pk2(b.x, b.y), X), r0, r1);
  return pack_h2(r0, r1);
}

// Key values of lower channels ch[0..3] (L: pairs (ch0, ch1), (ch2, ch3))
// and their partners (U) of token k of the lane's four (4gq + k), turned by
// R(4gq + k), as hi/lo A fragments (row rr of the A tile; [0] lower k-chunk,
// [1] partner k-chunk).  cs[h]: (cos, cos, sin, sin) of the pair h.  The turn
// and the hi/lo remainders run on packed fp32 pairs.
__device__ __forceinline__ void rope_key_frags(const float4 (&cs)[2], const uint64_t (&L)[2], const uint64_t (&U)[2],
                                               int rr, uint32_t (&ah)[2][4], uint32_t (&al)[2][4]) {
#pragma unroll
  for (int hp = 0; hp < 2; ++hp) {
    const uint64_t C = pk2(cs[hp].x, cs[hp].y), S = pk2(cs[hp].z, cs[hp].w);
    const uint64_t NL = sub2(mul2(L[hp], C), mul2(U[hp], S));  // l cos - u sin
    const uint64_t NU = fma2(L[hp], S, mul2(U[hp], C));        // l sin + u cos
    float l0, l1, u0, u1;
    upk2(NL, l0, l1);
    upk2(NU, u0, u1);
    const __half2 hl = __floats2half2_rn(l0, l1), hu = __floats2half2_rn(u0, u1);
    const float2 fl = __half22float2(hl), fu = __half22float2(hu);
    float dl0, dl1, du0, du1;
    upk2(sub2(NL, pk2(fl.x, fl.y)), dl0, dl1);
    upk2(sub2(NU, pk2(fu.x, fu.y)), du0, du1);
    ah[0][2 * hp + rr] = *reinterpret_cast<const uint32_t*>(&hl);
    al[0][2 * hp + rr] = pack_h2(dl0, dl1);
    ah[1][2 * hp + rr] = *reinterpret_cast<const uint32_t*>(&hu);
    al[1][2 * hp + rr] = pack_h2(du0, du1);
  }
}

// PV for one packed group: P^T per V block (probabilities times the per-token
// value scales), O^T += V^T P^T.
template <class C, class TR>
__device__ __forceinline__ void pv_packed(const Ctx<C>& cx, WarpState<C>& ws, const uint8_t* vsm, int n_valid,
                                          const float (&p)[C::NT][C::J][4]) {
  constexpr int D = C::D, NT = C::NT;
  const int gq = cx.gq, tq = cx.tq;
#pragma unroll
    for (int bv = 0; bv < D / TR::VG; ++bv) {
      uint32_t pb[2][NT][2], pbl[C::HC ? 2 : 1][NT][2];  // hi (or hi/lo columns), lo (heads as columns)
#pragma unroll
      for (int mu = 0; mu < 2; ++mu) {
        const int ra = 4 * gq + 2 * mu;
        const uint8_t* ha = vsm + ra * TR::VROW + bv * TR::VBB;
        const uint8_t* hb = ha + TR::VROW;
        const float sva = block_scale(ha);
        const float svb = block_scale(hb);
        float zpa = 0.f, zpb = 0.f;  // z' = z + beta s of rows a and b (asymmetric V)
        if constexpr (TR::Z) {
          zpa = fmaf(code_bias(TR::VB), sva, block_scale(ha + 2));
          zpb = fmaf(code_bias(TR::VB), svb, block_scale(hb + 2));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if constexpr (C::HC) {
            const float qa = ra < n_valid ? sva : 0.f, qb = ra + 1 < n_valid ? svb : 0.f;
            p_fragments_hc(p[nt][0][2 * mu] * qa, p[nt][1][2 * mu] * qa, pb[mu][nt][0], pbl[mu][nt][0]);
            p_fragments_hc(p[nt][0][2 * mu + 1] * qb, p[nt][1][2 * mu + 1] * qb, pb[mu][nt][1], pbl[mu][nt][1]);
          } else {
            const float pa = ra < n_valid ? p[nt][0][2 * mu] * sva : 0.f;
            const float pbb = ra + 1 < n_valid ? p[nt][0][2 * mu + 1] * svb : 0.f;
            p_fragments(pa, pbb, pb[mu][nt][0], pb[mu][nt][1]);
          }
          if constexpr (TR::Z) {
            const float za = ra < n_valid ? p[nt][0][2 * mu] * zpa : 0.f;
            const float zb = ra + 1 < n_valid ? p[nt][0][2 * mu + 1] * zpb : 0.f;
            ws.zo[bv][nt] += za + zb;
          }
        }
      }
#pragma unroll
      for (int ss = 0; ss < TR::VSPB; ++ss) {
        const int s = bv * TR::VSPB + ss;
        const int off = bv * TR::VBB + TR::HDR + ss * TR::VSPAN;
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          const int T1 = 8 * tq + 2 * mu;
          uint32_t x12[4], x34[4];
          if constexpr (TR::VB == 3) {
            static_assert(TR::VROW % 4 == 0 && C::VOFF % 4 == 0 && C::STAGE % 4 == 0, "4-byte aligned rows");
            v_pair4_3(vsm + T1 * TR::VROW, vsm + (T1 + 4) * TR::VROW, off, gq, x12);
            v_pair4_3(vsm + (T1 + 1) * TR::VROW, vsm + (T1 + 5) * TR::VROW, off, gq, x34);
          } else {
            v_pair4<TR, C::VSUB>(vsm + T1 * TR::VROW + off, vsm + (T1 + 4) * TR::VROW + off, gq, x12, cx.lut);
            v_pair4<TR, C::VSUB>(vsm + (T1 + 1) * TR::VROW + off, vsm + (T1 + 5) * TR::VROW + off, gq, x34,
                                 cx.lut);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(ws.o[2 * s][nt], x12[0], x12[1], x34[0], x34[1], pb[mu][nt][0], pb[mu][nt][1]);
            mma16816(ws.o[2 * s + 1][nt], x12[2], x12[3], x34[2], x34[3], pb[mu][nt][0], pb[mu][nt][1]);
            if constexpr (C::HC) {
              mma16816(ws.o[2 * s][nt], x12[0], x12[1], x34[0], x34[1], pbl[mu][nt][0], pbl[mu][nt][1]);
              mma16816(ws.o[2 * s + 1][nt], x12[2], x12[3], x34[2], x34[3], pbl[mu][nt][0], pbl[mu][nt][1]);
            }
            if constexpr (C::VSUB) {
              // the storage bias, removed in the same accumulator with every
              // group (rows: -beta 2^sh 2^-24 of their channel), so that o
              // never carries beta times the running probability sum
              constexpr uint32_t n0 = v_sub_neg(TR::VB, 0), n1 = v_sub_neg(TR::VB, 1);
              constexpr uint32_t n2 = v_sub_neg(TR::VB, 2), n3 = v_sub_neg(TR::VB, 3);
              mma16816(ws.o[2 * s][nt], n0, n1, n0, n1, pb[mu][nt][0], pb[mu][nt][1]);
              mma16816(ws.o[2 * s + 1][nt], n2, n3, n2, n3, pb[mu][nt][0], pb[mu][nt][1]);
              if constexpr (C::HC) {
                mma16816(ws.o[2 * s][nt], n0, n1, n0, n1, pbl[mu][nt][0], pbl[mu][nt][1]);
                mma16816(ws.o[2 * s + 1][nt], n2, n3, n2, n3, pbl[mu][nt][0], pbl[mu][nt][1]);
              }
            }
          }
        }
      }
    }
  }

// Scores of one packed group into S (see the layout notes at the top).
template <class C, class TR>
__device__ __forceinline__ void scores_packed(const Ctx<C>& cx, const uint8_t* ksm, int t0, float (&S)[2][C::NT][4]) {
  constexpr int D = C::D, NT = C::NT, KC = C::KC;
  const int gq = cx.gq, tq = cx.tq, lane = cx.lane;
  const uint32_t lo_mask = cx.lo_mask;
  const uint2* qb = cx.qb;
  const uint2* qh = cx.qh;
    if constexpr (TR::KCH && C::ROPE && !TR::Z) {
      // Pre-RoPE per-channel keys, t = t0 + j: with q' = R(-t0) q (fp32) and
      // codes c, scales s,
      //   q . R(t) k = sum_i cos(j th_i) (c_i s_i q'_i + c_u s_u q'_u)
      //                    + sin(j th_i) (c_i s_i q'_u - c_u s_u q'_i),  u = i + D/2.
      // The A operands are code x table entry, exact in fp16 (the table's hi
      // parts have 8 significant bits), for the hi and lo parts of cos and
      // sin; the B operands are the scaled, turned query in hi / lo columns.
      // Per k-chunk pair: 16 MMAs on two accumulator chains.
      const float2* base = cx.rope_base + (int64_t)(t0 / kTile) * (D / 2);
      const uint64_t NM = cx.lo_part ? pk2(-1.f, -1.f) : pk2(-0.f, -0.f);
      float Sx[2][NT][4];
#pragma unroll
      for (int mu = 0; mu < 2; ++mu)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Sx[mu][nt][0] = Sx[mu][nt][1] = Sx[mu][nt][2] = Sx[mu][nt][3] = 0.f;
#pragma unroll 1
      for (int kcp = 0; kcp < KC / 2; ++kcp) {
        float4 ql[NT], qu[NT];
        rope_query_f32<C>(cx, base, kcp, ql, qu);
        const int c = 32 * (kcp >> 1) + 8 * tq + 2 * (kcp & 1);
        const int ch[4] = {c, c + 4, c + 1, c + 5};
        float sl[4], su[4];
        uint32_t chl[4], chu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint8_t* bl = ksm + ch[q] * TR::KBB;
          const uint8_t* bu = ksm + (ch[q] + D / 2) * TR::KBB;
          sl[q] = block_scale(bl);
          su[q] = block_scale(bu);
          chl[q] = TR::KB == 4 ? ld_u16(bl + TR::HDR + 2 * gq) : (uint32_t)bl[TR::HDR + gq];
          chu[q] = TR::KB == 4 ? ld_u16(bu + TR::HDR + 2 * gq) : (uint32_t)bu[TR::HDR + gq];
        }
        // codes as exact fp16 pairs: [0] channels (c, c + 4), [1] (c + 1, c + 5), of token k
        uint32_t cl[2][4], cu[2][4];
        {
          const uint32_t xl0 = __byte_perm(chl[0], chl[1], 0x5410), xl1 = __byte_perm(chl[2], chl[3], 0x5410);
          const uint32_t xu0 = __byte_perm(chu[0], chu[1], 0x5410), xu1 = __byte_perm(chu[2], chu[3], 0x5410);
          if constexpr (TR::KB == 4) {
            dq4(xl0, cl[0]);
            dq4(xl1, cl[1]);
            dq4(xu0, cu[0]);
            dq4(xu1, cu[1]);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              cl[0][k] = code_pair<2>(xl0, k);
              cl[1][k] = code_pair<2>(xl1, k);
              cu[0][k] = code_pair<2>(xu0, k);
              cu[1][k] = code_pair<2>(xu1, k);
            }
          }
        }
        // B fragments of this lane's column (head gq / 2, hi or lo part)
        uint32_t bcl[NT][2], bsl[NT][2], bcu[NT][2], bsu[NT][2];
        const uint64_t L01 = pk2(sl[0], sl[1]), L23 = pk2(sl[2], sl[3]);
        const uint64_t U01 = pk2(su[0], su[1]), U23 = pk2(su[2], su[3]);
        const uint64_t N01 = pk2(-su[0], -su[1]), N23 = pk2(-su[2], -su[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint64_t a01 = pk2(ql[nt].x, ql[nt].y), a23 = pk2(ql[nt].z, ql[nt].w);
          const uint64_t b01 = pk2(qu[nt].x, qu[nt].y), b23 = pk2(qu[nt].z, qu[nt].w);
          bcl[nt][0] = col_pair(mul2(L01, a01), NM);
          bcl[nt][1] = col_pair(mul2(L23, a23), NM);
          bsl[nt][0] = col_pair(mul2(L01, b01), NM);
          bsl[nt][1] = col_pair(mul2(L23, b23), NM);
          bcu[nt][0] = col_pair(mul2(U01, b01), NM);
          bcu[nt][1] = col_pair(mul2(U23, b23), NM);
          bsu[nt][0] = col_pair(mul2(N01, a01), NM);
          bsu[nt][1] = col_pair(mul2(N23, a23), NM);
        }
        const uint4* tb = cx.rope_tab + (kcp * 4 * 2) * 32 + lane;  // [k][cos / sin][lane]
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          // turn table of the lane's tokens 2 mu (A rows gq) and 2 mu + 1 (rows gq + 8)
          const uint4 ca = __ldg(tb + (2 * mu) * 64), sa = __ldg(tb + (2 * mu) * 64 + 32);
          const uint4 cb = __ldg(tb + (2 * mu + 1) * 64), sb = __ldg(tb + (2 * mu + 1) * 64 + 32);
          const int ka = 2 * mu, kb = 2 * mu + 1;
#pragma unroll
          for (int side = 0; side < 2; ++side) {  // 0: lower channels, 1: partners
            const uint32_t(&x)[2][4] = side ? cu : cl;
            const uint32_t a_ch0 = hmul2u(x[0][ka], ca.x), a_ch1 = hmul2u(x[0][kb], cb.x);
            const uint32_t a_ch2 = hmul2u(x[1][ka], ca.y), a_ch3 = hmul2u(x[1][kb], cb.y);
            const uint32_t a_cl0 = hmul2u(x[0][ka], ca.z), a_cl1 = hmul2u(x[0][kb], cb.z);
            const uint32_t a_cl2 = hmul2u(x[1][ka], ca.w), a_cl3 = hmul2u(x[1][kb], cb.w);
            const uint32_t a_sh0 = hmul2u(x[0][ka], sa.x), a_sh1 = hmul2u(x[0][kb], sb.x);
            const uint32_t a_sh2 = hmul2u(x[1][ka], sa.y), a_sh3 = hmul2u(x[1][kb], sb.y);
            const uint32_t a_sl0 = hmul2u(x[0][ka], sa.z), a_sl1 = hmul2u(x[0][kb], sb.z);
            const uint32_t a_sl2 = hmul2u(x[1][ka], sa.w), a_sl3 = hmul2u(x[1][kb], sb.w);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint32_t(&bc)[2] = side ? bcu[nt] : bcl[nt];
              const uint32_t(&bs)[2] = side ? bsu[nt] : bsl[nt];
              mma16816(S[mu][nt], a_ch0, a_ch1, a_ch2, a_ch3, bc[0], bc[1]);
              mma16816(Sx[mu][nt], a_cl0, a_cl1, a_cl2, a_cl3, bc[0], bc[1]);
              mma16816(S[mu][nt], a_sh0, a_sh1, a_sh2, a_sh3, bs[0], bs[1]);
              mma16816(Sx[mu][nt], a_sl0, a_sl1, a_sl2, a_sl3, bs[0], bs[1]);
            }
          }
        }
      }
#pragma unroll
      for (int mu = 0; mu < 2; ++mu)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[mu][nt][e] += Sx[mu][nt][e];
    } else if constexpr (TR::KCH && C::ROPE) {
      // asymmetric blocks: each key value dequantized (with its zero point),
      // turned by R(j) in fp32 and split into fp16 hi + lo
      const float2* base = cx.rope_base + (int64_t)(t0 / kTile) * (D / 2);
#pragma unroll 1
      for (int kcp = 0; kcp < KC / 2; ++kcp) {
        uint32_t ql[NT][2], qu[NT][2];
        rope_query_pair<C>(cx, base, kcp, ql, qu);
        const int c = 32 * (kcp >> 1) + 8 * tq + 2 * (kcp & 1);
        const int ch[4] = {c, c + 4, c + 1, c + 5};
        float sl[4], su[4], zl[4] = {0.f, 0.f, 0.f, 0.f}, zu[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t xl[2], xu[2];
        uint32_t chl[4], chu[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint8_t* bl = ksm + ch[q] * TR::KBB;
          const uint8_t* bu = ksm + (ch[q] + D / 2) * TR::KBB;
          sl[q] = block_scale(bl);
          su[q] = block_scale(bu);
          if constexpr (TR::Z) {  // z' = z + beta s
            zl[q] = fmaf(code_bias(TR::KB), sl[q], block_scale(bl + 2));
            zu[q] = fmaf(code_bias(TR::KB), su[q], block_scale(bu + 2));
          }
          chl[q] = TR::KB == 4 ? ld_u16(bl + TR::HDR + 2 * gq) : (uint32_t)bl[TR::HDR + gq];
          chu[q] = TR::KB == 4 ? ld_u16(bu + TR::HDR + 2 * gq) : (uint32_t)bu[TR::HDR + gq];
        }
        xl[0] = __byte_perm(chl[0], chl[1], 0x5410);
        xl[1] = __byte_perm(chl[2], chl[3], 0x5410);
        xu[0] = __byte_perm(chu[0], chu[1], 0x5410);
        xu[1] = __byte_perm(chu[2], chu[3], 0x5410);
        uint32_t cl0[4], cl1[4], cu0[4], cu1[4];  // per token k of the thread: (ch0, ch1), (ch2, ch3)
        if constexpr (TR::KB == 4) {
          dq4(xl[0], cl0);
          dq4(xl[1], cl1);
          dq4(xu[0], cu0);
          dq4(xu[1], cu1);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            cl0[k] = code_pair<2>(xl[0], k);
            cl1[k] = code_pair<2>(xl[1], k);
            cu0[k] = code_pair<2>(xu[0], k);
            cu1[k] = code_pair<2>(xu[1], k);
          }
        }
        const float4* fr = cx.rope_frag + kcp * 256 + lane;
        // scales (and zeros) of the pairs (ch0, ch1), (ch2, ch3), lower and partner
        const uint64_t SL[2] = {pk2(sl[0], sl[1]), pk2(sl[2], sl[3])}, SU[2] = {pk2(su[0], su[1]), pk2(su[2], su[3])};
        const uint64_t ZL[2] = {pk2(zl[0], zl[1]), pk2(zl[2], zl[3])}, ZU[2] = {pk2(zu[0], zu[1]), pk2(zu[2], zu[3])};
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          uint32_t ah[2][4], al[2][4];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int k = 2 * mu + rr;
            const float4 cs[2] = {__ldg(fr + (2 * k) * 32), __ldg(fr + (2 * k + 1) * 32)};
            const float2 l01 = __half22float2(*reinterpret_cast<const __half2*>(&cl0[k]));
            const float2 l23 = __half22float2(*reinterpret_cast<const __half2*>(&cl1[k]));
            const float2 u01 = __half22float2(*reinterpret_cast<const __half2*>(&cu0[k]));
            const float2 u23 = __half22float2(*reinterpret_cast<const __half2*>(&cu1[k]));
            uint64_t Lv[2] = {pk2(l01.x, l01.y), pk2(l23.x, l23.y)}, Uv[2] = {pk2(u01.x, u01.y), pk2(u23.x, u23.y)};
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              Lv[hp] = TR::Z ? fma2(Lv[hp], SL[hp], ZL[hp]) : mul2(Lv[hp], SL[hp]);
              Uv[hp] = TR::Z ? fma2(Uv[hp], SU[hp], ZU[hp]) : mul2(Uv[hp], SU[hp]);
            }
            rope_key_frags(cs, Lv, Uv, rr, ah, al);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(S[mu][nt], ah[0][0], ah[0][1], ah[0][2], ah[0][3], ql[nt][0], ql[nt][1]);
            mma16816(S[mu][nt], al[0][0], al[0][1], al[0][2], al[0][3], ql[nt][0], ql[nt][1]);
            mma16816(S[mu][nt], ah[1][0], ah[1][1], ah[1][2], ah[1][3], qu[nt][0], qu[nt][1]);
            mma16816(S[mu][nt], al[1][0], al[1][1], al[1][2], al[1][3], qu[nt][0], qu[nt][1]);
          }
        }
      }
    } else if constexpr (TR::KCH) {
      // per-channel K: block c = channel c over the group's 32 tokens; the
      // channel scales multiply the query columns.  Even and odd k-chunks
      // accumulate separately (two independent MMA chains).  Codes are read
      // as subnormals (as v_pair4's), the token of a row fixing its position
      // factor; the bias comes off by one constant-row MMA per k-chunk, the
      // factors and 2^-24 once per group.  Asymmetric codes too: what remains
      // is field - beta, as the converted codes give, and the zero term below
      // adds z' = z + beta s.
      float Sx[2][NT][4];
#pragma unroll
      for (int mu = 0; mu < 2; ++mu)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) Sx[mu][nt][0] = Sx[mu][nt][1] = Sx[mu][nt][2] = Sx[mu][nt][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < KC; ++kc) {
        const int c = 32 * (kc >> 1) + 8 * tq + 2 * (kc & 1);
        const uint8_t* b1p = ksm + c * TR::KBB;
        const uint8_t* b2p = b1p + 4 * TR::KBB;
        const uint8_t* b3p = b1p + TR::KBB;
        const uint8_t* b4p = b1p + 5 * TR::KBB;
        uint32_t k12[4], k34[4];
        if constexpr (TR::KB == 4) {
          const uint32_t x12 = __byte_perm(ld_u16(b1p + TR::HDR + 2 * gq), ld_u16(b2p + TR::HDR + 2 * gq), 0x5410);
          const uint32_t x34 = __byte_perm(ld_u16(b3p + TR::HDR + 2 * gq), ld_u16(b4p + TR::HDR + 2 * gq), 0x5410);
          // token nibbles in place (positions 0, 4, 0, 4)
          k12[0] = x12 & 0x000F000Fu;
          k12[1] = x12 & 0x00F000F0u;
          k12[2] = (x12 >> 8) & 0x000F000Fu;
          k12[3] = (x12 >> 8) & 0x00F000F0u;
          k34[0] = x34 & 0x000F000Fu;
          k34[1] = x34 & 0x00F000F0u;
          k34[2] = (x34 >> 8) & 0x000F000Fu;
          k34[3] = (x34 >> 8) & 0x00F000F0u;
        } else {
          const uint32_t x12 = __byte_perm((uint32_t)b1p[TR::HDR + gq], (uint32_t)b2p[TR::HDR + gq], 0x5410);
          const uint32_t x34 = __byte_perm((uint32_t)b3p[TR::HDR + gq], (uint32_t)b4p[TR::HDR + gq], 0x5410);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // token fields in place (positions 0, 2, 4, 6)
            k12[k] = x12 & (0x00030003u << (2 * k));
            k34[k] = x34 & (0x00030003u << (2 * k));
          }
        }
        const uint32_t s12 = __byte_perm(ld_u16(b1p), ld_u16(b2p), 0x5410);
        const uint32_t s34 = __byte_perm(ld_u16(b3p), ld_u16(b4p), 0x5410);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          // q' * scale as fp16: hi = rn(q' s) on even columns, the exact
          // remainder fma(q', s, -hi) on odd columns (lo_mask all ones)
          const uint2 qv = qh[(kc * NT + nt) * 32 + lane];
          const uint32_t bq0 = hfma2u(qv.x, s12, (hmul2u(qv.x, s12) ^ 0x80008000u) & lo_mask);
          const uint32_t bq1 = hfma2u(qv.y, s34, (hmul2u(qv.y, s34) ^ 0x80008000u) & lo_mask);
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            float (&acc)[4] = (kc & 1) ? Sx[mu][nt] : S[mu][nt];
            mma16816(acc, k12[2 * mu], k12[2 * mu + 1], k34[2 * mu], k34[2 * mu + 1], bq0, bq1);
            // the storage bias of the rows' tokens, in the same accumulator
            const uint32_t na = v_sub_neg(TR::KB, 2 * mu), nb = v_sub_neg(TR::KB, 2 * mu + 1);
            mma16816(acc, na, nb, na, nb, bq0, bq1);
          }
        }
      }
#pragma unroll
      for (int mu = 0; mu < 2; ++mu)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            S[mu][nt][e] += Sx[mu][nt][e];
            // subnormal codes: rows gq / gq + 8 hold tokens 4 gq + 2 mu / + 1
            S[mu][nt][e] *= ldexpf(1.f, 24 - v_sub_shift(TR::KB, 2 * mu + (e >> 1)));
          }
      if constexpr (TR::Z) {
        // zero term of the group, the same for its 32 tokens: sum_c q'_c z'_c
        // with z'_c = z_c + beta s_c; lane l takes channels CPL l .. CPL l + CPL - 1
        constexpr int CPL = D / 32;
        static_assert(CPL % 4 == 0, "whole float4 query loads");
        float zq[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const uint8_t* blk = ksm + (CPL * lane + j) * TR::KBB;
          zq[j] = fmaf(code_bias(TR::KB), block_scale(blk), block_scale(blk + 2));
        }
        const int g = cx.g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float zs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int hl = 0; hl < 4; ++hl) {
            if (4 * nt + hl >= g) continue;  // warp-uniform
            const float* qrow = cx.qz + (4 * nt + hl) * D + CPL * lane;
            float acc = 0.f;
#pragma unroll
            for (int j4 = 0; j4 < CPL / 4; ++j4) {
              const float4 qv = *reinterpret_cast<const float4*>(qrow + 4 * j4);
              acc = fmaf(qv.x, zq[4 * j4], acc);
              acc = fmaf(qv.y, zq[4 * j4 + 1], acc);
              acc = fmaf(qv.z, zq[4 * j4 + 2], acc);
              acc = fmaf(qv.w, zq[4 * j4 + 3], acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            zs[hl] = acc;
          }
          // this lane's head is 4 nt + tq: add to its hi column (rows gq, gq + 8)
          const float zt = tq == 0 ? zs[0] : tq == 1 ? zs[1] : tq == 2 ? zs[2] : zs[3];
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            S[mu][nt][0] += zt;
            S[mu][nt][2] += zt;
          }
        }
      }
    } else {
      // per-token K: each K block's scale multiplies its partial scores
#pragma unroll
      for (int kb = 0; kb < D / TR::KG; ++kb) {
        float acc[2][NT][4];
#pragma unroll
        for (int mu = 0; mu < 2; ++mu)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) acc[mu][nt][0] = acc[mu][nt][1] = acc[mu][nt][2] = acc[mu][nt][3] = 0.f;
#pragma unroll
        for (int ss = 0; ss < TR::KSPB; ++ss) {
          const int s = kb * TR::KSPB + ss;
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            const int ra = 4 * gq + 2 * mu;
            uint32_t wa[4], wb[4];
            if constexpr (TR::KB == 3) {
              static_assert(TR::KROW % 4 == 0 && C::STAGE % 4 == 0, "4-byte aligned rows");
              const int off = kb * TR::KBB + TR::HDR + ss * TR::KSPAN;
              k_token_pairs3<C::KSUB>(ksm + ra * TR::KROW, off, tq, wa);
              k_token_pairs3<C::KSUB>(ksm + (ra + 1) * TR::KROW, off, tq, wb);
            } else {
              k_token_pairs<TR, C::KSUB>(ksm + ra * TR::KROW + kb * TR::KBB + TR::HDR + ss * TR::KSPAN, tq, wa,
                                         cx.lut);
              k_token_pairs<TR, C::KSUB>(ksm + (ra + 1) * TR::KROW + kb * TR::KBB + TR::HDR + ss * TR::KSPAN, tq, wb,
                                         cx.lut);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint2 q0 = qb[((2 * s) * NT + nt) * 32 + lane];
              const uint2 q1 = qb[((2 * s + 1) * NT + nt) * 32 + lane];
              mma16816(acc[mu][nt], wa[0], wb[0], wa[1], wb[1], q0.x, q0.y);
              mma16816(acc[mu][nt], wa[2], wb[2], wa[3], wb[3], q1.x, q1.y);
              if constexpr (C::HC) {  // the query's lo parts, same accumulator
                const uint2 r0 = cx.qbl[((2 * s) * NT + nt) * 32 + lane];
                const uint2 r1 = cx.qbl[((2 * s + 1) * NT + nt) * 32 + lane];
                mma16816(acc[mu][nt], wa[0], wb[0], wa[1], wb[1], r0.x, r0.y);
                mma16816(acc[mu][nt], wa[2], wb[2], wa[3], wb[3], r1.x, r1.y);
              }
            }
          }
        }
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          const float sa = block_scale(ksm + (4 * gq + 2 * mu) * TR::KROW + kb * TR::KBB);
          const float sb = block_scale(ksm + (4 * gq + 2 * mu + 1) * TR::KROW + kb * TR::KBB);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if constexpr (C::KSUB) {
              // subnormal codes: (2^24 acc - beta sum of the column's query) s
              const float2 kq = reinterpret_cast<const float2*>(cx.kq)[(kb * NT + nt) * 4 + tq];
              const float ua = sa * 0x1p24f, ub = sb * 0x1p24f;
              S[mu][nt][0] = fmaf(acc[mu][nt][0], ua, fmaf(-kq.x, sa, S[mu][nt][0]));
              S[mu][nt][1] = fmaf(acc[mu][nt][1], ua, fmaf(-kq.y, sa, S[mu][nt][1]));
              S[mu][nt][2] = fmaf(acc[mu][nt][2], ub, fmaf(-kq.x, sb, S[mu][nt][2]));
              S[mu][nt][3] = fmaf(acc[mu][nt][3], ub, fmaf(-kq.y, sb, S[mu][nt][3]));
            } else {
              S[mu][nt][0] += acc[mu][nt][0] * sa;
              S[mu][nt][1] += acc[mu][nt][1] * sa;
              S[mu][nt][2] += acc[mu][nt][2] * sb;
              S[mu][nt][3] += acc[mu][nt][3] * sb;
            }
          }
        }
      }
    }
  }

// Chunked token splits.  The grid holds n_units x splits blocks (the block
// budget), spread over the units by tile count rather than evenly per unit:
// every unit of n tiles is cut into ceil(n / C) nearly equal chunks (a unit
// with no tiles into one empty chunk), C the smallest chunk of at least min_chunk
// tiles (and of the longest unit / kMaxSplits; of the longest unit / splits
// when the caller fixed the count) whose chunks fit the grid.  Uniform
// lengths give every unit `splits` chunks, as an even split would; in a
// ragged batch long sequences get more chunks and short ones fewer, so every
// block carries about the same number of tiles.  Blocks are numbered
// unit-major (layer, sequence, kv head, chunk): a unit's chunks, and so its
// partial rows, are consecutive.  Blocks past the last chunk have no work.
// Warp 0 plans from every sequence's length (batches of up to kChunkSeqs
// sequences; larger ones, one block per unit, grids of more than two waves
// of resident blocks and batches of equal lengths split evenly).
constexpr int kChunkSeqs = 256;

struct Work {
  int li, seq, h, T, chunk, n_chunks, tb, te, first;  // first: linear index of the unit's chunk 0
  int active, bad_len;
};

// Tiles of a unit of T tokens (cold, hot / main, window; the first two 32-token
// groups, the window in 32-token tiles).
template <bool HAS_COLD>
__device__ __forceinline__ int unit_tiles(const Layout& lo, int T) {
  const int qe = q_end_of(lo, T);
  const int ce = HAS_COLD ? c_end_of(lo, T) : 0;
  return ce / kTile + (qe - ce + kTile - 1) / kTile + (T - qe + kTile - 1) / kTile;
}

// n / C rounded down and up, for 0 <= n < 2^22 and C >= 1 (tile counts), with
// rc = 1/C in fp32: n rc lies within n/C 2^-23 <= 1/2 of n / C, so its
// truncation is off by at most one, which one exact step corrects.
__device__ __forceinline__ int floor_div_tiles(int n, int C, float rc) {
  int q = (int)__fmul_rn((float)n, rc);
  if (q * C > n) --q;
  else if ((q + 1) * C <= n) ++q;
  return q;
}
__device__ __forceinline__ int ceil_div_tiles(int n, int C, float rc) {
  const int q = floor_div_tiles(n, C, rc);
  return q + (q * C < n ? 1 : 0);
}

// The attended length of sequence s (0, flagged by the caller, when outside
// [0, max_T]).
__device__ __forceinline__ int attended_len(const DecodeArgs& a, int s, int* bad) {
  const int T = a.seq_lens[s] + a.len_add;
  if (T < 0 || T > a.lo.max_T) {
    *bad = 1;
    return 0;
  }
  *bad = 0;
  return T;
}

// This block's work (all threads call it; one __syncthreads inside).
template <bool HAS_COLD>
__device__ __forceinline__ Work plan_work(const DecodeArgs& a, Work* sw) {
  const Layout& lo = a.lo;
  const int B = lo.B, H = lo.H, S = a.splits, k = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    Work w{};
    // even split of every unit: one block per unit, one sequence, a
    // multi-wave grid (the block scheduler balances it), batches too large to
    // plan, or (found below) equal tile counts
    bool even = S == 1 || B == 1 || !a.chunked || B > kChunkSeqs || lo.max_T >= (1 << 26);
    constexpr int kPer = kChunkSeqs / 32;
    int n[kPer], bad[kPer], T[kPer], maxn = 0, minn = 0x7FFFFFFF, sum = 0;
    // lane l holds sequences [l per, (l + 1) per)
    const int per = (B + 31) / 32, s0 = lane * per;
    if (!even) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        n[j] = 0;
        bad[j] = 0;
        T[j] = 0;
        if (j < per && s0 + j < B) {
          T[j] = attended_len(a, s0 + j, &bad[j]);
          n[j] = unit_tiles<HAS_COLD>(lo, T[j]);
          maxn = max(maxn, n[j]);
          minn = min(minn, n[j]);
          sum += n[j];
        }
      }
      maxn = __reduce_max_sync(0xFFFFFFFFu, maxn);
      minn = __reduce_min_sync(0xFFFFFFFFu, minn);
      even = maxn == minn && !a.fixed_splits;
    }
    if (even) {
      // the unit's share of the budget: the grid's S blocks, or fewer when
      // the grid was widened for a budget that is not a multiple of B
      const int nc = max(1, min(S, a.budget / B));
      const int unit = k / S;
      w.chunk = k % S;
      w.n_chunks = nc;
      w.first = unit * S;
      w.h = unit % H;
      w.seq = (unit / H) % B;
      w.li = unit / (H * B);
      w.active = w.li < a.n_layers && w.chunk < nc;
      if (w.active) {
        w.T = attended_len(a, w.seq, &w.bad_len);
        const int n = unit_tiles<HAS_COLD>(lo, w.T);
        w.tb = (int)((int64_t)w.chunk * n / nc);
        w.te = (int)((int64_t)(w.chunk + 1) * n / nc);
      }
      if (lane == 0) *sw = w;
    } else {
      const int N = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)sum), K = a.budget;  // one layer's kv head
      int c_lo = max(max(a.min_chunk, 1), (maxn + kMaxSplits - 1) / kMaxSplits);
      if (a.fixed_splits) c_lo = max(c_lo, (maxn + S - 1) / S);
      // the smallest C >= c_lo with chunks(C) <= K: chunks(C) >= N / C, and
      // chunks(C) < N / C + B, so it lies in [N / K, N / (K - B)] (K > B: the
      // host gives a budget of at least 2 B when S > 1), and C = maxn gives B
      // chunks
      auto chunks = [&](int C) {
        const float rc = __frcp_rn((float)C);
        int c = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j)
          if (j < per && s0 + j < B) c += max(1, ceil_div_tiles(n[j], C, rc));
        return (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)c);
      };
      int c_hi = max(c_lo, min(maxn, (N + K - B - 1) / (K - B)));
      c_lo = min(c_hi, max(c_lo, (N + K - 1) / K));
      while (c_lo < c_hi) {
        const int mid = c_lo + (c_hi - c_lo) / 2;
        if (chunks(mid) <= K) c_hi = mid;
        else c_lo = mid + 1;
      }
      const int C = c_lo;
      const float rc = __frcp_rn((float)C);
      int nch[kPer], mine = 0;  // chunks per sequence; this lane's, times H (one layer)
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        nch[j] = (j < per && s0 + j < B) ? max(1, ceil_div_tiles(n[j], C, rc)) : 0;
        mine += H * nch[j];
      }
      int incl = mine;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += y;
      }
      const int P = __shfl_sync(0xFFFFFFFFu, incl, 31);  // blocks per layer
      const int li = k / P, r = k - li * P;
      if (li >= a.n_layers) {
        if (lane == 0) *sw = w;  // inactive
      } else if (r >= incl - mine && r < incl) {  // exactly one lane
        int base = incl - mine;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          if (j < per && s0 + j < B) {
            const int nc = nch[j];
            if (r < base + H * nc) {
              const int o = r - base;
              w.li = li;
              w.seq = s0 + j;
              w.h = floor_div_tiles(o, nc, __frcp_rn((float)nc));
              w.chunk = o - w.h * nc;
              w.n_chunks = nc;
              w.first = k - w.chunk;
              w.T = T[j];
              w.bad_len = bad[j];
              // the unit's tiles in nc nearly equal chunks (at most C each)
              w.tb = (int)((int64_t)w.chunk * n[j] / nc);
              w.te = (int)((int64_t)(w.chunk + 1) * n[j] / nc);
              w.active = 1;
              *sw = w;
              break;
            }
            base += H * nc;
          }
        }
      }
    }
  }
  __syncthreads();
  return *sw;
}

// Fused decode step: the append of this step's token for the tiles it changes
// that lie in this block's range [tb, te) (tiles after the step: cold, hot /
// main, window).  The token changes at most three tiles: the group that moves
// from hot to cold (phase A), the unit that moves from the window into the
// packed tier (phase B) and the window slot of the token itself (phase C).
// Each tile belongs to exactly one block, which writes it before decoding it,
// and no block reads a tile it does not own, so no block waits for another.
// The step for per-token 128-value blocks without a window (the rotated
// layouts): the new token is quantized at once.  Warp w takes chunk w of the
// token (K chunks, then V chunks), lane l its values 4l..4l+3: the same
// randomized transform as the append kernels, the block's absolute maximum,
// the fp16 scale, and code = clamp(rint(x / s)) with the IEEE quotient, packed
// in the format's bit fields (4 bits: nibbles, value i in byte i / 2; 3 bits:
// a little-endian stream, 8 values per 24-bit word).
template <int NC>
__device__ __forceinline__ void step_token128(const AppendArgs& s, int li, int seq, int h, int t) {
  const Layout& lo = s.lo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int layer = s.layer0 + li;
  for (int item = warp; item < 2 * NC; item += kWarps) {
    const int which = item / NC, c = item % NC;
    const FmtInfo& f = fmt_main(lo, which);
    const uint16_t* src = (which ? s.v : s.k) + (((int64_t)li * s.total_new + seq) * lo.H + h) * lo.D + 128 * c;
    const float4 x = f16x4_to_f32(*reinterpret_cast<const uint2*>(src + 4 * lane), lo.dtype);
    float v[4] = {x.x, x.y, x.z, x.w};
    if (lo.flags & (which ? KVQ_ROTATE_V : KVQ_ROTATE_K)) warp_rotate128(v, lo.d1, lo.d2);
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const __half s16 = block_scale_of(m, f.qmax);
    const float sf = __half2float(s16);
    const int bias = 1 << (f.bits - 1);
    uint32_t fld = 0;  // this lane's 4 biased codes, f.bits bits each
#pragma unroll
    for (int e = 0; e < 4; ++e) fld |= (uint32_t)(quant_code(v[e], sf, f.qmax) + bias) << (f.bits * e);
    const uint32_t nxt = __shfl_down_sync(0xffffffffu, fld, 1);
    bool bad = false;
    uint8_t* blk = main_row(lo, s.cp, which, layer, seq, h, t, &bad);
    if (bad) {  // warp-uniform
      if (lane == 0) atomicOr(s.status, KVQ_DEV_PAGE);
      continue;
    }
    blk += c * f.bb;
    if (lane == 0) *reinterpret_cast<__half*>(blk) = s16;
    if (f.bits == 4) {
      *reinterpret_cast<uint16_t*>(blk + 2 + 2 * lane) = (uint16_t)fld;
    } else if ((lane & 1) == 0) {  // 3 bits: lanes 2m, 2m + 1 form the 24-bit word m
      const uint32_t w24 = fld | (nxt << 12);
      uint8_t* p = blk + 2 + 3 * (lane >> 1);
      p[0] = (uint8_t)w24;
      p[1] = (uint8_t)(w24 >> 8);
      p[2] = (uint8_t)(w24 >> 16);
    }
  }
}

// The generic append phases of the step, out of line: inlined, they push
// the decode loop out of the instruction cache.
template <int NC>
__device__ __noinline__ void step_phase_a(const AppendArgs& s, int li, int seq, int h) {
  append_requant_unit<NC>(s, li, seq, h, 0);
}
template <int NC>
__device__ __noinline__ void step_phase_b(const AppendArgs& s, int li, int seq, int h, uint8_t* sm) {
  append_quantize_unit<NC, false>(s, li, seq, h, 0, sm);
}
__device__ __noinline__ void step_phase_c(const AppendArgs& s, int li, int seq, int h) {
  append_window_unit(s, li, seq, h, 0);
}

template <class C, bool ROT>
__device__ __forceinline__ void step_append(const DecodeArgs& a, const Work& w, uint8_t* sm) {
  const Layout& lo = a.lo;
  const int T = w.T, T0 = T - 1;  // attended length T0 + 1 (one new token)
  if (!w.active || w.bad_len || T0 < 0) return;  // flagged by the decode
  const int h = w.h, li = w.li, seq = w.seq, tb = w.tb, te = w.te;
  const int qe = q_end_of(lo, T);
  const int ce = C::HAS_COLD ? c_end_of(lo, T) : 0;
  const int n_c = ce / kTile;
  const int n_m = (qe - ce + kTile - 1) / kTile;
  const int q0 = q_end_of(lo, T0);
  const int c0 = C::HAS_COLD ? c_end_of(lo, T0) : 0;
  auto mine = [&](int tile) { return tile >= tb && tile < te; };
  if constexpr (ROT) {  // per-token 128-value blocks, no window: the token itself, in tile T0 / 32
    if (mine(T0 / kTile)) step_token128<C::D / 128>(a.step, li, seq, h, T0);
    return;
  }
  if (C::HAS_COLD && ce > c0 && mine(n_c - 1)) step_phase_a<C::D / 128>(a.step, li, seq, h);
  if (qe > q0 && mine(q0 < ce ? q0 / kTile : n_c + (q0 - ce) / kTile)) step_phase_b<C::D / 128>(a.step, li, seq, h, sm);
  if (T0 >= qe && mine(n_c + n_m + (T0 - qe) / kTile)) step_phase_c(a.step, li, seq, h);
}

// Shared-memory scratch of the step's generic phase B (raw rows); the
// 128-value path needs none.
template <class C, bool ROT>
constexpr int step_smem() {
  return ROT ? 0 : 2 * kTile * (C::D + 8) * 2;
}

// STEP: 0 decode only; 1 fused decode step through the generic append
// phases (windows, tiers, per-channel groups); 2 fused decode step of
// per-token 128-value blocks without a window (step_token128).
template <class C, int STEP>
__global__ void __launch_bounds__(kThreadsMma, C::MIN_CTAS) decode_mma_kernel(DecodeArgs a) {
  constexpr int D = C::D, NT = C::NT, KC = C::KC;
  extern __shared__ __align__(16) uint8_t smem[];
  // launched with programmatic stream serialization: wait for the previous
  // grid of the stream (and its memory) before reading anything, and let the
  // next grid's blocks become resident as soon as this grid's blocks leave
  grid_dependency_wait();
  grid_launch_dependents();
  uint2* qb = reinterpret_cast<uint2*>(smem);  // [KC][NT][32 lanes]: this lane's B fragment (b0, b1)
  uint2* qh = qb + KC * NT * 32;               // [KC][NT][32 lanes]: query half pairs (per-channel K)
  float4* qr = reinterpret_cast<float4*>(qh + (C::QH ? KC * NT * 32 : 0));  // [KC][NT][32]: fp32 query (RoPE)
  float* qz = reinterpret_cast<float*>(qr + (C::ROPE ? KC * NT * 32 : 0));  // [4 NT][D] (asymmetric K)
  uint2* qbl = reinterpret_cast<uint2*>(qz + (C::Z ? 4 * NT * D : 0));     // [KC][NT][32 lanes]: lo (HC)
  float* kq = reinterpret_cast<float*>(qbl + (C::HC ? KC * NT * 32 : 0));  // [KBLK][NT][8] (KSUB)
  uint8_t* stage_base = smem + C::QSM;
  __shared__ float qmax_s[kWarps];
  __shared__ uint32_t bad_page;
  constexpr int kStages = C::STAGES;
  __shared__ uint64_t mbar[kWarps * kMaxStages];
  __shared__ uint64_t never_bar;  // no thread ever arrives on it (failure-detection test mode)
  __shared__ int is_last;
  __shared__ int pf_page[kWarps][2][2];  // paged: next tile's page ids per warp, by issue parity
  __shared__ Work work_s;
  __shared__ const uint8_t* lin[2];  // K and V addresses of cold tile 0 (tiered) or page 0 (paged)
  __shared__ int pstride[2];         // paged: bytes from one page of this (layer, kv head) to the next

  // the plan stays in shared memory: its fields are read where needed, not
  // held in registers across the group loop
  (void)plan_work<C::HAS_COLD>(a, &work_s);
  const Work& w = work_s;
  if (!w.active) return;
  if constexpr (STEP != 0) {
    // the step's cache writes first, then this block's decode reads them:
    // generic-proxy writes ordered before the bulk copies (async proxy)
    step_append<C, STEP == 2>(a, w, smem);
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
    __syncthreads();
  }
  const Layout& lo = a.lo;
  const int g = lo.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int h = w.h, li = w.li, seq = w.seq, tb = w.tb, te = w.te, T = w.T;
  const int layer = a.layer0 + li;
  const int tid = threadIdx.x;
  if (w.bad_len && w.chunk == 0 && h == 0 && tid == 0) atomicOr(a.status, KVQ_DEV_LENGTH);
  const int qe = q_end_of(lo, T);
  const int ce = C::HAS_COLD ? c_end_of(lo, T) : 0;
  const int n_c = ce / kTile;
  const int n_m = (qe - ce + kTile - 1) / kTile;
  const int64_t qrow = ((int64_t)li * lo.B + seq) * lo.Hq + (int64_t)h * g;

  // ---- barriers, then the first bulk copies: they land while the query is prepared ----
  if (tid == 0) {
    bad_page = 0;
    if constexpr (C::HAS_COLD) {
      lin[0] = cold_row(lo, a.cp, 0, layer, seq, h, 0);
      lin[1] = cold_row(lo, a.cp, 1, layer, seq, h, 0);
    } else if (lo.paged) {
      const int64_t r0 = ((int64_t)layer * lo.n_pages * lo.H + h) * lo.pt;  // page 0's first row
      lin[0] = a.cp.k_main + r0 * lo.kf.row;
      lin[1] = a.cp.v_main + r0 * lo.vf.row;
      pstride[0] = lo.H * lo.pt * lo.kf.row;
      pstride[1] = lo.H * lo.pt * lo.vf.row;
    }
  }
  if (tid < kWarps * kStages) mbar_init(mbar + tid, 1);
  if (tid == kThreadsMma - 1) mbar_init(&never_bar, 1);
  fence_mbar_init();
  // (the step's scratch rows in shared memory were written through the
  // generic proxy: order them before the bulk copies into the same bytes)
  fence_proxy_async();
  __syncthreads();
  uint8_t* wst = stage_base + warp * kStages * C::STAGE;

  // Paged tiles: lane 0 copies the page ids of the next tile it will issue
  // into shared memory (4-byte cp.async) one issue ahead, so the block-table
  // reads overlap a group of compute instead of stalling the copy issue; no
  // register holds them across the loop.
  const int first = tb + warp;  // this warp takes tiles first, first + kWarps, ...

  // Cold tiles, and the tiles of an untiered contiguous main tier, lie one
  // tile stride apart: tile t of this unit starts t strides after tile 0.
  // Tile 0's K and V addresses sit in shared memory (lin[0], lin[1]) for the
  // tiered kernels, whose registers are fuller, and in lane 0's registers
  // (k_lin, v_lin) otherwise.  (The hot ring looks each tile's rows up.)
  // Pages: page p of this (layer, kv head) starts p page strides (pstride)
  // after page 0, whose addresses lin then holds.
  const uint8_t* k_lin = nullptr;
  const uint8_t* v_lin = nullptr;
  if constexpr (!C::HAS_COLD) {
    if (lane == 0 && !lo.paged && !lo.tiered) {
      bool unused = false;
      k_lin = main_row(lo, a.cp, 0, layer, seq, h, 0, &unused);
      v_lin = main_row(lo, a.cp, 1, layer, seq, h, 0, &unused);
    }
  }

  // Bulk copies of packed tile `tile` (cold or hot/only tier) into stage
  // `st`, issued by lane 0: exactly one arrival on the stage's barrier per
  // packed tile of this warp (with no bytes when a page id is bad).
  auto issue = [&](int tile, int st) {
    if (tile >= te || tile >= n_c + n_m) return;
    if (lane != 0) return;
    uint8_t* ks = wst + st * C::STAGE;
    uint8_t* vs = ks + C::VOFF;
    uint64_t* bar = mbar + warp * kStages + st;
    if constexpr (C::HAS_COLD) {
      if (tile < n_c) {
        const uint8_t* kg = lin[0] + (int64_t)tile * C::COLD::KSTAGE;
        const uint8_t* vg = lin[1] + (int64_t)tile * C::COLD::VSTAGE;
        if (!(span_ok(lo, a.cp, 2, kg, C::COLD::KSTAGE) & span_ok(lo, a.cp, 3, vg, C::COLD::VSTAGE))) {
          mbar_arrive_tx(bar, 0);  // bounds-checked build only: skipped
          return;
        }
        mbar_arrive_tx(bar, C::COLD::KSTAGE + C::COLD::VSTAGE);
        bulk_g2s(ks, kg, C::COLD::KSTAGE, bar);
        bulk_g2s(vs, vg, C::COLD::VSTAGE, bar);
        return;
      }
    }
    using HT = typename C::HOT;
    const int t0 = ce + (tile - n_c) * kTile;
    bool bad = false;
    if (lo.paged) {
      // one or two pages (16-token pages when the group is complete); tiles
      // start at multiples of 32, so at row 0 of a page
      const int np = (qe - t0 > lo.pt) ? kTile / lo.pt : 1;
      const int kb = lo.pt * HT::KROW, vb = lo.pt * HT::VROW;
      // this warp issues tiles first, first + kWarps, ...: the ids of every
      // tile after the first were copied by the issue before it
      const int par = ((tile - first) / kWarps) & 1;
      const int* bt_row = a.cp.block_table + (int64_t)seq * lo.max_pages;
      int p0, p1;
      if (tile == first || (tile - kWarps) < n_c) {
        p0 = bt_row[t0 / lo.pt];
        p1 = np == 2 ? bt_row[t0 / lo.pt + 1] : p0;
      } else {
        cp_async_wait<0>();
        p0 = pf_page[warp][par][0];
        p1 = np == 2 ? pf_page[warp][par][1] : p0;
      }
      const int nx = tile + kWarps;  // the next tile this warp issues
      if (nx < te && nx >= n_c && nx < n_c + n_m) {
        const int pn = (ce + (nx - n_c) * kTile) / lo.pt;
        cp_async4(&pf_page[warp][par ^ 1][0], bt_row + pn);
        cp_async4(&pf_page[warp][par ^ 1][1], bt_row + pn + (qe - pn * lo.pt > lo.pt ? 1 : 0));
        cp_async_commit();
      }
      if (p0 < 0 || p0 >= lo.n_pages || p1 < 0 || p1 >= lo.n_pages) {
        bad_page = 1;
        mbar_arrive_tx(bar, 0);
        return;
      }
      const uint8_t* k0 = lin[0] + (int64_t)p0 * pstride[0];
      const uint8_t* v0 = lin[1] + (int64_t)p0 * pstride[1];
      const uint8_t* k1 = lin[0] + (int64_t)p1 * pstride[0];
      const uint8_t* v1 = lin[1] + (int64_t)p1 * pstride[1];
      if (!(span_ok(lo, a.cp, 0, k0, kb) & span_ok(lo, a.cp, 1, v0, vb) & span_ok(lo, a.cp, 0, k1, kb) &
            span_ok(lo, a.cp, 1, v1, vb))) {
        mbar_arrive_tx(bar, 0);  // bounds-checked build only: skipped
        return;
      }
      mbar_arrive_tx(bar, np * (kb + vb));
      bulk_g2s(ks, k0, kb, bar);
      bulk_g2s(vs, v0, vb, bar);
      if (np == 2) {
        bulk_g2s(ks + kb, k1, kb, bar);
        bulk_g2s(vs + vb, v1, vb, bar);
      }
      return;
    }
    const uint8_t* kg = k_lin ? k_lin + (int64_t)tile * HT::KSTAGE : main_row(lo, a.cp, 0, layer, seq, h, t0, &bad);
    const uint8_t* vg = k_lin ? v_lin + (int64_t)tile * HT::VSTAGE : main_row(lo, a.cp, 1, layer, seq, h, t0, &bad);
    if (!(span_ok(lo, a.cp, 0, kg, HT::KSTAGE) & span_ok(lo, a.cp, 1, vg, HT::VSTAGE))) {
      mbar_arrive_tx(bar, 0);  // bounds-checked build only: skipped
      return;
    }
    mbar_arrive_tx(bar, HT::KSTAGE + HT::VSTAGE);
    bulk_g2s(ks, kg, HT::KSTAGE, bar);
    bulk_g2s(vs, vg, HT::VSTAGE, bar);
  };

  // the query scratch takes the last QSLOTS stage slots of the last warp,
  // which that warp fills only after the query is prepared
  constexpr int QSLOTS = ((C::HC ? 8 : 4 * NT) * D * 4 + C::STAGE - 1) / C::STAGE;
  static_assert(QSLOTS <= kStages, "query scratch fits in the last warp's stage slots");
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i)
    if (warp != kWarps - 1 || i < kStages - QSLOTS) issue(first + kWarps * i, i);

  // ---- query: fp32, rotated when K is stored rotated; per-lane fragments ----
  float qexp = 1.f;
  {
    float* qf = reinterpret_cast<float*>(stage_base + (kWarps * kStages - QSLOTS) * C::STAGE);  // [g][D]
    for (int e = tid; e < g * D; e += kThreadsMma) qf[e] = in_to_f32(a.q[qrow * D + e], lo.dtype);
    __syncthreads();
    if (lo.flags & KVQ_ROTATE_K) {
      for (int r = warp; r < g * (D / 128); r += kWarps) {
        float* p = qf + r * 128 + 4 * lane;
        float v[4] = {p[0], p[1], p[2], p[3]};
        warp_rotate128(v, lo.d1, lo.d2);
        p[0] = v[0];
        p[1] = v[1];
        p[2] = v[2];
        p[3] = v[3];
      }
      __syncthreads();
    }
    // power-of-two normalization: |q'| = |q| 2^-e <= 1, so products with fp16
    // scales cannot overflow fp16 (the factor 2^e returns with the score scale)
    float m = 0.f;
    for (int e = tid; e < g * D; e += kThreadsMma) m = fmaxf(m, fabsf(qf[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) qmax_s[warp] = m;
    __syncthreads();
    m = fmaxf(fmaxf(qmax_s[0], qmax_s[1]), fmaxf(qmax_s[2], qmax_s[3]));
    int ex = 0;
    if (m > 0.f) frexpf(m, &ex);
    // pre-RoPE keys: one more halving, so the turned query (|q'| < sqrt(2))
    // times an fp16 scale stays below 65504
    if constexpr (C::ROPE) ex += 1;
    const float qnorm = ldexpf(1.f, -ex);
    qexp = ldexpf(1.f, ex);
    for (int e = tid; e < KC * NT * 32; e += kThreadsMma) {
      const int ln = e & 31, nt = (e >> 5) % NT, kc = (e >> 5) / NT;
      const int c = 32 * (kc >> 1) + 8 * (ln & 3) + 2 * (kc & 1);
      // column ln / 4: head 8 nt + column (heads as columns, hi fragment here)
      // or head 4 nt + column / 2, hi / lo by the column's parity
      const int hh = C::HC ? 8 * nt + (ln >> 2) : 4 * nt + ((ln >> 2) >> 1);
      const bool lo = !C::HC && ((ln >> 2) & 1) != 0;
      float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
      if (hh < g) {
        const float* q = qf + hh * D;
        v0 = q[c] * qnorm;
        v1 = q[c + 4] * qnorm;
        v2 = q[c + 1] * qnorm;
        v3 = q[c + 5] * qnorm;
        if constexpr (C::KSUB) {  // the codes' position factors, taken out of the query (exact)
          const float f0 = ldexpf(1.f, -k_sub_shift(C::HOT::KB, kc & 1, false));
          const float f1 = ldexpf(1.f, -k_sub_shift(C::HOT::KB, kc & 1, true));
          v0 *= f0;
          v1 *= f0;
          v2 *= f1;
          v3 *= f1;
        }
      }
      qb[e] = make_uint2(pack_h2(split_part(v0, lo), split_part(v1, lo)),
                         pack_h2(split_part(v2, lo), split_part(v3, lo)));
      if constexpr (C::HC)
        qbl[e] = make_uint2(pack_h2(split_part(v0, true), split_part(v1, true)),
                            pack_h2(split_part(v2, true), split_part(v3, true)));
      if constexpr (C::QH) qh[e] = make_uint2(pack_h2(v0, v1), pack_h2(v2, v3));
      if constexpr (C::ROPE) qr[e] = make_float4(v0, v1, v2, v3);
    }
    if constexpr (C::Z) {
      for (int e = tid; e < 4 * NT * D; e += kThreadsMma) {
        const int hh = e / D;
        qz[e] = hh < g ? qf[e] * qnorm : 0.f;
      }
    }
    if constexpr (C::KSUB) {
      // beta times the sum, over each K block's channels, of the fp16 values
      // each column's MMAs multiply (the fragments times their position
      // factors; hi and lo fragments with heads as columns)
      __syncthreads();
      constexpr int CPB = KC / C::KBLK;  // k-chunks per K block
      for (int e = tid; e < C::KBLK * NT * 8; e += kThreadsMma) {
        const int col = e & 7, nt = (e >> 3) % NT, kb = (e >> 3) / NT;
        float sum = 0.f;
        for (int kc = kb * CPB; kc < (kb + 1) * CPB; ++kc) {
          const float f0 = ldexpf(1.f, k_sub_shift(C::HOT::KB, kc & 1, false));
          const float f1 = ldexpf(1.f, k_sub_shift(C::HOT::KB, kc & 1, true));
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int i = (kc * NT + nt) * 32 + 4 * col + t;
            uint2 fr[2] = {qb[i], C::HC ? qbl[i] : make_uint2(0u, 0u)};
#pragma unroll
            for (int u = 0; u < (C::HC ? 2 : 1); ++u) {
              const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&fr[u].x));
              const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&fr[u].y));
              sum += f0 * (x.x + x.y) + f1 * (y.x + y.y);
            }
          }
        }
        kq[e] = (float)k_sub_bias(C::HOT::KB) * sum;
      }
    }
    __syncthreads();
  }
  const bool lo_part = (gq & 1) != 0;
  const uint32_t lo_mask = lo_part ? 0xFFFFFFFFu : 0u;
  const float qscale = kLog2eF / sqrtf((float)D) * qexp;
  Ctx<C> cx;
  cx.gq = gq;
  cx.tq = tq;
  cx.lane = lane;
  cx.lo_part = lo_part;
  cx.lo_mask = lo_mask;
  cx.qb = qb;
  cx.qbl = qbl;
  cx.qh = qh;
  cx.qr = qr;
  cx.qz = qz;
  cx.kq = kq;
  cx.g = g;
  cx.rope_base = a.rope;
  cx.rope_frag = reinterpret_cast<const float4*>(a.rope + (int64_t)(a.rope_base_rows + kTile) * (D / 2));
  cx.rope_tab = reinterpret_cast<const uint4*>(a.rope + (int64_t)(a.rope_base_rows + 2 * kTile) * (D / 2));
  if constexpr (C::HOT::KLUT || C::HOT::VLUT) {
    uint32_t m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = __half_as_ushort(__float2half_rn(lo.cb[8 + k]));  // exact: fp16 entries
    cx.lut[0] = (m[0] & 0xFF) | (m[1] & 0xFF) << 8 | (m[2] & 0xFF) << 16 | (m[3] & 0xFF) << 24;
    cx.lut[1] = (m[4] & 0xFF) | (m[5] & 0xFF) << 8 | (m[6] & 0xFF) << 16 | (m[7] & 0xFF) << 24;
    cx.lut[2] = (m[0] >> 8) | (m[1] >> 8) << 8 | (m[2] >> 8) << 16 | (m[3] >> 8) << 24;
    cx.lut[3] = (m[4] >> 8) | (m[5] >> 8) << 8 | (m[6] >> 8) << 16 | (m[7] >> 8) << 24;
  } else {
    cx.lut[0] = cx.lut[1] = cx.lut[2] = cx.lut[3] = 0;
  }

  WarpState<C> ws;
#pragma unroll
  for (int i = 0; i < KC; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) ws.o[i][nt][e] = 0.f;
#pragma unroll
  for (int i = 0; i < NT * C::J; ++i) {
    ws.m[i] = -INFINITY;
    ws.l[i] = 0.f;
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int s = 0; s < (C::Z ? C::NS : 1); ++s) ws.zo[s][nt] = 0.f;

  }
  // ---- per-warp pipeline over this CTA's groups --------------------------------
  // the query scratch was written through the generic proxy: order it before
  // the bulk copies into those slots (the last warp's deferred ones, the loop's)
  fence_proxy_async();
  __syncthreads();
  if (warp == kWarps - 1) {
#pragma unroll
    for (int i = kStages - QSLOTS; i < kStages - 1; ++i) issue(first + kWarps * i, i);
  }
  int stall_it = -1;
  bool vsub_done = false;  // subnormal V: o is in plain units
  for (int it = 0;; ++it) {
    const int tile = first + kWarps * it;
    if (tile >= te) break;
    issue(tile + kWarps * (kStages - 1), (it + kStages - 1) % kStages);
    if (tile < n_c + n_m) {
      // test mode: the first wait is on a barrier nothing completes, bounded
      // by a.stall_polls polls, so the stall path below runs for real
      const bool landed = (a.stall_polls > 0 && it == 0)
                              ? mbar_wait(&never_bar, 0, a.stall_polls)
                              : mbar_wait(mbar + warp * kStages + it % kStages, (it / kStages) & 1);
      if (!landed) {
        stall_it = it;
        break;
      }
    }

    float S[2][NT][4];
#pragma unroll
    for (int mu = 0; mu < 2; ++mu)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) S[mu][nt][0] = S[mu][nt][1] = S[mu][nt][2] = S[mu][nt][3] = 0.f;
    float p[NT][C::J][4];

    if (tile < n_c + n_m) {
      // ---------------- packed group from shared memory ----------------
      const uint8_t* ksm = wst + (it % kStages) * C::STAGE;
      const uint8_t* vsm = ksm + C::VOFF;
      bool cold = false;
      if constexpr (C::HAS_COLD) cold = tile < n_c;
      if (cold) {
        if constexpr (C::HAS_COLD) {
          const int t0 = tile * kTile;
          scores_packed<C, typename C::COLD>(cx, ksm, t0, S);
          online_softmax<C>(ws, S, kTile, gq, qscale, p);
          pv_packed<C, typename C::COLD>(cx, ws, vsm, kTile, p);
        }
      } else {
        const int t0 = ce + (tile - n_c) * kTile;
        const int n_valid = min(kTile, qe - t0);
        scores_packed<C, typename C::HOT>(cx, ksm, t0, S);
        online_softmax<C>(ws, S, n_valid, gq, qscale, p);
        pv_packed<C, typename C::HOT>(cx, ws, vsm, n_valid, p);
      }
    } else {
      // ---------------- 16-bit window group from global memory ----------------
      if (!vsub_done) {  // a warp's window groups come after all its packed groups
        vsub_finish<C>(ws);
        vsub_done = true;
      }
      const int t0 = qe + (tile - n_c - n_m) * kTile;
      const int n_valid = min(kTile, T - t0);
      if constexpr (C::ROPE) {
        const float2* base = cx.rope_base + (int64_t)(t0 / kTile) * (D / 2);
#pragma unroll 1
        for (int kcp = 0; kcp < KC / 2; ++kcp) {
          uint32_t ql[NT][2], qu[NT][2];
          rope_query_pair<C>(cx, base, kcp, ql, qu);
          // k-chunk kcp: channels c + {0, 4, 1, 5}, c = 32 (kcp / 2) + 8 tq + 2 (kcp % 2)
          const int c = 32 * (kcp >> 1) + 8 * tq + 2 * (kcp & 1);
          const float4* fr = cx.rope_frag + kcp * 256 + lane;
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            uint32_t ah[2][4], al[2][4];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int k = 2 * mu + rr, r = 4 * gq + k;
              const uint16_t* row = resid_row(lo, a.cp, 0, layer, seq, h, t0 + min(r, n_valid - 1));
              uint32_t wl0 = 0, wl1 = 0, wu0 = 0, wu1 = 0;  // (c, c+1), (c+4, c+5) and partners
              if (r < n_valid) {
                wl0 = *reinterpret_cast<const uint32_t*>(row + c);
                wl1 = *reinterpret_cast<const uint32_t*>(row + c + 4);
                wu0 = *reinterpret_cast<const uint32_t*>(row + c + D / 2);
                wu1 = *reinterpret_cast<const uint32_t*>(row + c + 4 + D / 2);
              }
              const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&wl0));
              const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&wl1));
              const float2 b0 = __half22float2(*reinterpret_cast<const __half2*>(&wu0));
              const float2 b1 = __half22float2(*reinterpret_cast<const __half2*>(&wu1));
              const uint64_t Lv[2] = {pk2(a0.x, a1.x), pk2(a0.y, a1.y)}, Uv[2] = {pk2(b0.x, b1.x), pk2(b0.y, b1.y)};
              const float4 cs[2] = {__ldg(fr + (2 * k) * 32), __ldg(fr + (2 * k + 1) * 32)};
              rope_key_frags(cs, Lv, Uv, rr, ah, al);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(S[mu][nt], ah[0][0], ah[0][1], ah[0][2], ah[0][3], ql[nt][0], ql[nt][1]);
              mma16816(S[mu][nt], al[0][0], al[0][1], al[0][2], al[0][3], ql[nt][0], ql[nt][1]);
              mma16816(S[mu][nt], ah[1][0], ah[1][1], ah[1][2], ah[1][3], qu[nt][0], qu[nt][1]);
              mma16816(S[mu][nt], al[1][0], al[1][1], al[1][2], al[1][3], qu[nt][0], qu[nt][1]);
            }
          }
        }
      } else {
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          const int ra = 4 * gq + 2 * mu, rb = ra + 1;
          const uint16_t* rowa = resid_row(lo, a.cp, 0, layer, seq, h, t0 + min(ra, n_valid - 1));
          const uint16_t* rowb = resid_row(lo, a.cp, 0, layer, seq, h, t0 + min(rb, n_valid - 1));
#pragma unroll
          for (int s = 0; s < C::NS; ++s) {
            uint4 va = make_uint4(0, 0, 0, 0), vb = va;
            if (ra < n_valid) va = *reinterpret_cast<const uint4*>(rowa + 32 * s + 8 * tq);
            if (rb < n_valid) vb = *reinterpret_cast<const uint4*>(rowb + 32 * s + 8 * tq);
            // pairs (c, c+4), (c+1, c+5), (c+2, c+6), (c+3, c+7)
            const uint32_t a0 = __byte_perm(va.x, va.z, 0x5410), a1 = __byte_perm(va.x, va.z, 0x7632);
            const uint32_t a2 = __byte_perm(va.y, va.w, 0x5410), a3 = __byte_perm(va.y, va.w, 0x7632);
            const uint32_t b0 = __byte_perm(vb.x, vb.z, 0x5410), b1 = __byte_perm(vb.x, vb.z, 0x7632);
            const uint32_t b2 = __byte_perm(vb.y, vb.w, 0x5410), b3 = __byte_perm(vb.y, vb.w, 0x7632);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              uint2 q0 = qb[((2 * s) * NT + nt) * 32 + lane];
              uint2 q1 = qb[((2 * s + 1) * NT + nt) * 32 + lane];
              uint2 r0, r1;
              if constexpr (C::HC) {
                r0 = cx.qbl[((2 * s) * NT + nt) * 32 + lane];
                r1 = cx.qbl[((2 * s + 1) * NT + nt) * 32 + lane];
              }
              if constexpr (C::KSUB) {
                // 16-bit keys carry no position factors: put them back into
                // the query fragments (powers of two)
                q0 = unsub_frag<C::HOT::KB, false>(q0);
                q1 = unsub_frag<C::HOT::KB, true>(q1);
                if constexpr (C::HC) {
                  r0 = unsub_frag<C::HOT::KB, false>(r0);
                  r1 = unsub_frag<C::HOT::KB, true>(r1);
                }
              }
              mma16816(S[mu][nt], a0, b0, a1, b1, q0.x, q0.y);
              mma16816(S[mu][nt], a2, b2, a3, b3, q1.x, q1.y);
              if constexpr (C::HC) {
                mma16816(S[mu][nt], a0, b0, a1, b1, r0.x, r0.y);
                mma16816(S[mu][nt], a2, b2, a3, b3, r1.x, r1.y);
              }
            }
          }
        }
      }
      online_softmax<C>(ws, S, n_valid, gq, qscale, p);
      uint32_t pb[2][NT][2], pbl[C::HC ? 2 : 1][NT][2];
#pragma unroll
      for (int mu = 0; mu < 2; ++mu) {
        const int ra = 4 * gq + 2 * mu;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float va = ra < n_valid ? 1.f : 0.f, vb = ra + 1 < n_valid ? 1.f : 0.f;
          if constexpr (C::HC) {
            p_fragments_hc(p[nt][0][2 * mu] * va, p[nt][1][2 * mu] * va, pb[mu][nt][0], pbl[mu][nt][0]);
            p_fragments_hc(p[nt][0][2 * mu + 1] * vb, p[nt][1][2 * mu + 1] * vb, pb[mu][nt][1], pbl[mu][nt][1]);
          } else {
            p_fragments(p[nt][0][2 * mu] * va, p[nt][0][2 * mu + 1] * vb, pb[mu][nt][0], pb[mu][nt][1]);
          }
        }
      }
#pragma unroll
      for (int mu = 0; mu < 2; ++mu) {
        const int T1 = 8 * tq + 2 * mu;
        const int tk[4] = {T1, T1 + 4, T1 + 1, T1 + 5};
        const uint16_t* rows[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) rows[k] = resid_row(lo, a.cp, 1, layer, seq, h, t0 + min(tk[k], n_valid - 1));
#pragma unroll
        for (int s = 0; s < C::NS; ++s) {
          uint2 r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            r[k] = make_uint2(0, 0);
            if (tk[k] < n_valid) r[k] = *reinterpret_cast<const uint2*>(rows[k] + 32 * s + 4 * gq);
          }
          // (token pair, channel 4gq+j) halves
          const uint32_t x0 = __byte_perm(r[0].x, r[1].x, 0x5410), x1 = __byte_perm(r[0].x, r[1].x, 0x7632);
          const uint32_t x2 = __byte_perm(r[0].y, r[1].y, 0x5410), x3 = __byte_perm(r[0].y, r[1].y, 0x7632);
          const uint32_t y0 = __byte_perm(r[2].x, r[3].x, 0x5410), y1 = __byte_perm(r[2].x, r[3].x, 0x7632);
          const uint32_t y2 = __byte_perm(r[2].y, r[3].y, 0x5410), y3 = __byte_perm(r[2].y, r[3].y, 0x7632);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(ws.o[2 * s][nt], x0, x1, y0, y1, pb[mu][nt][0], pb[mu][nt][1]);
            mma16816(ws.o[2 * s + 1][nt], x2, x3, y2, y3, pb[mu][nt][0], pb[mu][nt][1]);
            if constexpr (C::HC) {
              mma16816(ws.o[2 * s][nt], x0, x1, y0, y1, pbl[mu][nt][0], pbl[mu][nt][1]);
              mma16816(ws.o[2 * s + 1][nt], x2, x3, y2, y3, pbl[mu][nt][0], pbl[mu][nt][1]);
            }
          }
        }
      }
    }
    // every lane is done with this stage before lane 0 refills it
    fence_proxy_async();
    __syncwarp();
  }
  if (!vsub_done) vsub_finish<C>(ws);
  if (lo.paged && lane == 0) cp_async_wait<0>();  // a page-id copy issued for a tile not reached
  if (stall_it >= 0) {
    // a copy did not land in time: flag it, give this warp's copies still in
    // flight (that tile's and the next one's) a last bounded wait, and merge
    // whatever is there
    if (lane == 0) atomicOr(a.status, KVQ_DEV_STALL);
    for (int j = stall_it; j < stall_it + kStages; ++j) {
      const int tj = first + kWarps * j;
      if (tj < te && tj < n_c + n_m) (void)mbar_wait(mbar + warp * kStages + j % kStages, (j / kStages) & 1);
    }
  }
  __syncthreads();

  // ---- merge the warps (shared memory), then the splits (workspace) -------------
  float* wm = reinterpret_cast<float*>(stage_base);  // [kWarps][g]
  float* wl = wm + kWarps * kMaxGqa;                  // [kWarps][g]
  float* wo = wl + kWarps * kMaxGqa;                  // [kWarps][g][D]
  float* obuf = wo + kWarps * kMaxGqa * D;            // [g][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float zo[C::Z ? C::NS : 1] = {};  // zero-point part of the output per 32-channel block
    if constexpr (C::Z) {
#pragma unroll
      for (int s = 0; s < C::NS; ++s) {
        float z = ws.zo[s][nt];
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 8);
        z += __shfl_xor_sync(0xffffffffu, z, 16);
        zo[s] = z;
      }
    }
#pragma unroll
    for (int j = 0; j < C::J; ++j) {
      float l = ws.l[nt * C::J + j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int hh = C::HC ? 8 * nt + 2 * tq + j : 4 * nt + tq;
      if (hh < g) {
        if (gq == 0) {
          wm[warp * kMaxGqa + hh] = ws.m[nt * C::J + j];
          wl[warp * kMaxGqa + hh] = l;
        }
        float* orow = wo + (warp * kMaxGqa + hh) * D;
#pragma unroll
        for (int s = 0; s < C::NS; ++s)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ch = 32 * s + 4 * gq + 2 * e;
            if constexpr (C::HC) {  // column 2tq + j of rows gq, gq + 8
              orow[ch] = ws.o[2 * s + e][nt][j];
              orow[ch + 1] = ws.o[2 * s + e][nt][2 + j];
            } else {  // hi + lo columns
              const float zadd = C::Z ? zo[C::Z ? s : 0] : 0.f;
              orow[ch] = ws.o[2 * s + e][nt][0] + ws.o[2 * s + e][nt][1] + zadd;
              orow[ch + 1] = ws.o[2 * s + e][nt][2] + ws.o[2 * s + e][nt][3] + zadd;
            }
          }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && bad_page) atomicOr(a.status, KVQ_DEV_PAGE);
  // CTA partial per head: M = max_w m_w, L = sum_w 2^(m_w - M) l_w, O likewise
  const int64_t unit = ((int64_t)li * lo.B + seq) * lo.H + h;
  constexpr int PR = part_row(D);
  float* part = a.partials + (int64_t)(w.first + w.chunk) * g * PR;
  for (int e = tid; e < g * D; e += kThreadsMma) {
    const int hh = e / D, d = e % D;
    float M = -INFINITY;
    for (int wi = 0; wi < kWarps; ++wi) M = fmaxf(M, wm[wi * kMaxGqa + hh]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int wi = 0; wi < kWarps; ++wi) {
        const float sc = exp2f(wm[wi * kMaxGqa + hh] - M);
        L += sc * wl[wi * kMaxGqa + hh];
        O += sc * wo[(wi * kMaxGqa + hh) * D + d];
      }
    }
    if (w.n_chunks == 1) {
      obuf[e] = L > 0.f ? O / L : 0.f;
    } else {
      part[hh * PR + d] = O;
      if (d == 0) {
        part[hh * PR + D] = M;
        part[hh * PR + D + 1] = L;
      }
    }
  }
  if (w.n_chunks > 1) {
    // two levels when the unit has at least 4 kCombineFan chunks: the last
    // chunk of each group of kCombineFan merges the group into the group's
    // first row, then the last group merges the group rows (one level below
    // that: two serial merges cost more than one longer merge)
    constexpr int F = kCombineFan;
    uint32_t* tk = a.tickets + unit * kTicketsPerUnit;  // [0]: the unit, [1 + group]: its groups
    float* rows = a.partials + (int64_t)w.first * g * PR;
    const int n_grp = w.n_chunks >= 4 * F ? (w.n_chunks + F - 1) / F : 1, grp = w.chunk / F, g0 = grp * F;
    const int gn = min(F, w.n_chunks - g0);
    // the per-warp partials in wo are dead here: the merge weights reuse them
    static_assert(kWarps * kMaxGqa * D >= kMaxGqa * kMaxSplits, "merge weights fit in the warp partials");
    __threadfence();
    __syncthreads();
    if (n_grp > 1 && gn > 1) {
      if (tid == 0) is_last = atomicAdd(tk + 1 + grp, 1u) == (unsigned)(gn - 1);
      __syncthreads();
      if (!is_last) return;
      __threadfence();
      float* grow = rows + (int64_t)g0 * g * PR;
      combine_rows<D, kThreadsMma, false>(grow, gn, 1, g, grow, wo, wm);
      if (tid == 0) tk[1 + grp] = 0;
      __threadfence();
      __syncthreads();
    }
    const int n_last = n_grp > 1 ? n_grp : w.n_chunks;  // rows of the final merge
    if (tid == 0) is_last = atomicAdd(tk, 1u) == (unsigned)(n_last - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    combine_rows<D, kThreadsMma, true>(rows, n_last, n_grp > 1 ? F : 1, g, obuf, wo, wm);
    if (tid == 0) tk[0] = 0;
  }
  __syncthreads();
  if (lo.flags & KVQ_ROTATE_V) {
    for (int r = warp; r < g * (D / 128); r += kWarps) {
      float* pp = obuf + r * 128 + 4 * lane;
      float v[4] = {pp[0], pp[1], pp[2], pp[3]};
      warp_unrotate128(v, lo.d1, lo.d2);
      pp[0] = v[0];
      pp[1] = v[1];
      pp[2] = v[2];
      pp[3] = v[3];
    }
    __syncthreads();
  }
  for (int e = tid; e < g * D; e += kThreadsMma) a.out[qrow * D + e] = obuf[e];
}

template <class C, int STEP>
cudaError_t launch_mma(const DecodeArgs& a, cudaStream_t st) {
  static_assert(C::SMEM >= C::QSM + (2 * kWarps * kMaxGqa + kWarps * kMaxGqa * C::D + kMaxGqa * C::D) * 4,
                "merge scratch must fit in the stage buffers");
  constexpr int smem = STEP != 0 && step_smem<C, STEP == 2>() > C::SMEM ? step_smem<C, STEP == 2>() : C::SMEM;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<C, STEP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_dependent(decode_mma_kernel<C, STEP>, dim3(a.splits * a.lo.H * a.n_layers * a.lo.B),
                          dim3(kThreadsMma), smem, st, a);
}

bool fmt_is(const FmtInfo& f, int bits, int group, int axis) {
  return f.bits == bits && f.group == group && f.axis == axis;
}

template <int D, int KF, int KG, int VF, int VG, bool Z = false>
using T_ = Tier<D, KF, KG, VF, VG, Z>;

// Whether the tensor-core kernel takes this cache at all (layout limits).
inline bool mma_layout_ok(const Layout& lo) {
  bool ok = true;
  if (lo.ring) ok = ok && lo.dtype == KVQ_DT_F16 && !(lo.flags & (KVQ_ROTATE_K | KVQ_ROTATE_V));
  if (lo.paged) ok = ok && (lo.pt == 16 || lo.pt == 32);
  if (lo.kf.codebook != lo.vf.codebook) ok = false;  // one tensor TBQ4, the other not: generic kernel
  if (lo.kf.zp != lo.vf.zp) ok = false;              // one tensor asymmetric, the other not: generic kernel
  return ok;
}

}  // namespace
}  // namespace kvq
