// Split-K decode attention on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulators) for single-tier caches:
//   K per-channel 4-bit over 32-token groups, or per-token 8/4/3-bit blocks;
//   V per-token 8/4/3-bit blocks; an optional fp16 window; optional rotation
//   (no window then); contiguous or 16/32-token pages.
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
// Layout of one group: M-tile mu (0, 1) row r is token
// tau(mu, r) = 4(r & 7) + 2mu + (r >> 3); k-chunk kc = 2s + b (span s of 32
// channels) pairs channels (c, c+4) in k-slots (2t, 2t+1) and (c+1, c+5) in
// (2t+8, 2t+9), c = 32s + 8t + 2b (t = lane % 4); d-tile (s, e) row r is
// channel 32s + 4(r & 7) + 2e + (r >> 3).
//
// Work split: CTA = 4 warps on one (layer, sequence, kv head, token split);
// each warp streams its own groups through a 3-stage cp.async ring and keeps
// its own online softmax; warps merge in shared memory and splits merge in
// the workspace (the last CTA to take a ticket combines; nobody waits).
#include "block_codec.cuh"

namespace kvq {

cudaError_t launch_decode_generic(const DecodeArgs& a, cudaStream_t s);

namespace {

enum : int { KF_CH4 = 0, KF_T8 = 1, KF_T4 = 2, KF_T3 = 3 };
enum : int { VF_T8 = 0, VF_T4 = 1, VF_T3 = 2 };

constexpr int kWarps = 4;
constexpr int kThreadsMma = kWarps * 32;
constexpr int kStages = 3;
constexpr float kLog2eF = 1.4426950408889634f;

constexpr int bits_k(int kf) { return kf == KF_T8 ? 8 : kf == KF_T3 ? 3 : 4; }
constexpr int bits_v(int vf) { return vf == VF_T8 ? 8 : vf == VF_T3 ? 3 : 4; }
constexpr int align16(int x) { return (x + 15) / 16 * 16; }

template <int D_, int NT_, int KF_, int KG_, int VF_, int VG_>
struct Cfg {
  static constexpr int D = D_, NT = NT_, KF = KF_, KG = KG_, VF = VF_, VG = VG_;
  static constexpr int KB = bits_k(KF), VB = bits_v(VF);
  static constexpr bool KCH = KF == KF_CH4;
  static constexpr int KBB = 2 + (KCH ? 32 : KG) * KB / 8;  // block bytes
  static constexpr int VBB = 2 + VG * VB / 8;
  static constexpr int KROW = KCH ? D * KBB : (D / KG) * KBB;  // group row / token row
  static constexpr int VROW = (D / VG) * VBB;
  static constexpr int KSTAGE = KCH ? KROW : 32 * KROW;
  static constexpr int VSTAGE = 32 * VROW;
  static constexpr int VOFF = align16(KSTAGE + 16);
  static constexpr int STAGE = VOFF + align16(VSTAGE + 16);
  static constexpr int KC = D / 16;  // k-chunks
  static constexpr int NS = D / 32;  // spans
  static constexpr int KSPB = KCH ? 1 : KG / 32;  // spans per K block
  static constexpr int VSPB = VG / 32;
  static constexpr int KSPAN = 32 * KB / 8;  // code bytes of a span of one token
  static constexpr int VSPAN = 32 * VB / 8;
  static constexpr int QSM = KC * NT * 32 * 16;  // per-lane query values
  static constexpr int SMEM = QSM + kWarps * kStages * STAGE;
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

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }
// four bytes at an even address
__device__ __forceinline__ uint32_t ld_u32e(const uint8_t* p) { return ld_u16(p) | (ld_u16(p + 2) << 16); }
// 24 bits at any byte address (reads the aligned word after it too)
__device__ __forceinline__ uint32_t ld_u24(const uint8_t* p) {
  const uintptr_t ad = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(ad & ~uintptr_t(3));
  return __funnelshift_r(w[0], w[1], (uint32_t)(ad & 3) * 8) & 0xFFFFFFu;
}

// Two codes of B bits at bit B*j of each 16-bit half of x, as an exact fp16
// pair (code with the storage bias removed).
template <int B>
__device__ __forceinline__ uint32_t code_pair(uint32_t x, int j) {
  if constexpr (B == 4) return hsub2u(((x >> (4 * j)) & 0x000F000Fu) | 0x64006400u, 0x64086408u);
  if constexpr (B == 3) return hsub2u(((x >> (3 * j)) & 0x00070007u) | 0x64006400u, 0x64046404u);
  return hsub2u(((x >> (2 * j)) & 0x00030003u) | 0x64006400u, 0x64026402u);
}
// Two int8 codes in byte 0 of each 16-bit half of (x >> 8j).
__device__ __forceinline__ uint32_t code_pair8(uint32_t x, int j) {
  return hsub2u(((x >> (8 * j)) & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}

// Eight K codes (channels c0..c0+7 of one token) as four fp16 pairs
// (c0+j, c0+j+4), j = 0..3.  `p` points at the first code byte of the span.
template <class C>
__device__ __forceinline__ void k_token_pairs(const uint8_t* p, int tq, uint32_t (&r)[4]) {
  if constexpr (C::KB == 4) {
    const uint32_t w = ld_u32e(p + 4 * tq);
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = code_pair<4>(w, j);
  } else if constexpr (C::KB == 8) {
    const uint32_t w0 = ld_u32e(p + 8 * tq), w1 = ld_u32e(p + 8 * tq + 4);
    const uint32_t xa = __byte_perm(w0, w1, 0x5410), xb = __byte_perm(w0, w1, 0x7632);
    r[0] = code_pair8(xa, 0);
    r[1] = code_pair8(xa, 1);
    r[2] = code_pair8(xb, 0);
    r[3] = code_pair8(xb, 1);
  } else {  // 3 bits, 8 codes in 24 bits
    const uint32_t w = ld_u24(p + 3 * tq);
    const uint32_t x = (w & 0xFFFu) | ((w << 4) & 0x0FFF0000u);
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = code_pair<3>(x, j);
  }
}

// Four V codes (channels 4*gq..4*gq+3 of a span) of token rows ra and rb as
// four fp16 pairs (row a, row b) for channel 4gq+j.  p* point at the span's
// first code byte of each row.
template <class C>
__device__ __forceinline__ void v_pair4(const uint8_t* pa, const uint8_t* pb, int gq, uint32_t (&r)[4]) {
  if constexpr (C::VB == 8) {
    const uint32_t wa = ld_u32e(pa + 4 * gq), wb = ld_u32e(pb + 4 * gq);
    const uint32_t xa = __byte_perm(wa, wb, 0x5410), xb = __byte_perm(wa, wb, 0x7632);
    r[0] = code_pair8(xa, 0);
    r[1] = code_pair8(xa, 1);
    r[2] = code_pair8(xb, 0);
    r[3] = code_pair8(xb, 1);
  } else {
    uint32_t ua, ub;
    if constexpr (C::VB == 4) {
      ua = ld_u16(pa + 2 * gq);
      ub = ld_u16(pb + 2 * gq);
    } else {  // 3 bits: 12 bits at bit 12*gq of the span
      const int sh = 12 * (gq & 1), bo = 3 * (gq >> 1);
      ua = (ld_u24(pa + bo) >> sh) & 0xFFFu;
      ub = (ld_u24(pb + bo) >> sh) & 0xFFFu;
    }
    const uint32_t x = ua | (ub << 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = code_pair<C::VB>(x, j);
  }
}

template <class C>
struct WarpState {
  float o[C::KC][C::NT][4];
  float m[C::NT], l[C::NT];
};

// Online softmax over one group's scores; returns the probabilities of the
// thread's four tokens 4gq..4gq+3 for each n-tile.
template <class C>
__device__ __forceinline__ void online_softmax(WarpState<C>& ws, float (&S)[2][C::NT][4], int n_valid, int gq,
                                               float qscale, float (&p)[C::NT][4]) {
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt) {
    float s[4];
    s[0] = (S[0][nt][0] + S[0][nt][1]) * qscale;
    s[1] = (S[0][nt][2] + S[0][nt][3]) * qscale;
    s[2] = (S[1][nt][0] + S[1][nt][1]) * qscale;
    s[3] = (S[1][nt][2] + S[1][nt][3]) * qscale;
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (4 * gq + k >= n_valid) s[k] = -INFINITY;
      mx = fmaxf(mx, s[k]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(ws.m[nt], mx);
    const float alpha = exp2f(ws.m[nt] - m_new);
    ws.m[nt] = m_new;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      p[nt][k] = exp2f(s[k] - m_new);
      sum += p[nt][k];
    }
    ws.l[nt] = ws.l[nt] * alpha + sum;
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int i = 0; i < C::KC; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) ws.o[i][nt][e] *= alpha;
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

template <class C>
__global__ void __launch_bounds__(kThreadsMma) decode_mma_kernel(DecodeArgs a) {
  constexpr int D = C::D, NT = C::NT;
  extern __shared__ __align__(16) uint8_t smem[];
  float4* qsm = reinterpret_cast<float4*>(smem);  // [KC][NT][32 lanes]
  uint8_t* stage_base = smem + C::QSM;
  __shared__ uint32_t bad_page;
  __shared__ int is_last;

  const Layout& lo = a.lo;
  const int g = lo.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y;
  const int li = blockIdx.z / lo.B, seq = blockIdx.z % lo.B;
  const int layer = a.layer0 + li;
  const int tid = threadIdx.x;

  int T = a.seq_lens[seq];
  if (T < 0 || T > lo.max_T) {
    if (split == 0 && h == 0 && tid == 0) atomicOr(a.status, KVQ_DEV_LENGTH);
    T = 0;
  }
  const int qe = q_end_of(lo, T);
  const int n_m = (qe + kTile - 1) / kTile;
  const int n_w = (T - qe + kTile - 1) / kTile;
  const int ntiles = n_m + n_w;
  const int tb = (int)((int64_t)split * ntiles / a.splits);
  const int te = (int)((int64_t)(split + 1) * ntiles / a.splits);
  const int64_t qrow = ((int64_t)li * lo.B + seq) * lo.Hq + (int64_t)h * g;

  // ---- query: fp32, rotated when K is stored rotated; per-lane values -------
  {
    float* qf = reinterpret_cast<float*>(stage_base);  // [g][D] scratch
    for (int e = tid; e < g * D; e += kThreadsMma) qf[e] = in_to_f32(a.q[qrow * D + e], lo.dtype);
    if (tid == 0) bad_page = 0;
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
    for (int e = tid; e < C::KC * NT * 32; e += kThreadsMma) {
      const int ln = e & 31, nt = (e >> 5) % NT, kc = (e >> 5) / NT;
      const int c = 32 * (kc >> 1) + 8 * (ln & 3) + 2 * (kc & 1);
      const int hh = 4 * nt + ((ln >> 2) >> 1);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (hh < g) {
        const float* qr = qf + hh * D;
        v = make_float4(qr[c], qr[c + 4], qr[c + 1], qr[c + 5]);
      }
      qsm[e] = v;
    }
    __syncthreads();
  }
  const bool lo_part = (gq & 1) != 0;
  const float qscale = kLog2eF / sqrtf((float)D);

  WarpState<C> ws;
#pragma unroll
  for (int i = 0; i < C::KC; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) ws.o[i][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    ws.m[nt] = -INFINITY;
    ws.l[nt] = 0.f;
  }
  uint8_t* wst = stage_base + warp * kStages * C::STAGE;

  // query fragment (b0, b1) of k-chunk kc, n-tile nt, unscaled (hi or lo part)
  auto qfrag = [&](int kc, int nt, uint32_t& b0, uint32_t& b1) {
    const float4 v = qsm[(kc * NT + nt) * 32 + lane];
    b0 = pack_h2(split_part(v.x, lo_part), split_part(v.y, lo_part));
    b1 = pack_h2(split_part(v.z, lo_part), split_part(v.w, lo_part));
  };

  // copies of main-tier tile `tile` into stage `st` (nothing for window tiles)
  auto issue = [&](int tile, int st) {
    if (tile >= te || tile >= n_m) return;
    const int t0 = tile * kTile;
    uint8_t* ks = wst + st * C::STAGE;
    uint8_t* vs = ks + C::VOFF;
    bool bad = false;
    if (lo.paged) {
      const int np = (qe - t0 > lo.pt) ? kTile / lo.pt : 1;
      const int kb = lo.pt * C::KROW, vb = lo.pt * C::VROW;
      for (int pg = 0; pg < np; ++pg) {
        const uint8_t* kg = main_row(lo, a.cp, 0, layer, seq, h, t0 + pg * lo.pt, &bad);
        const uint8_t* vg = main_row(lo, a.cp, 1, layer, seq, h, t0 + pg * lo.pt, &bad);
        if (bad) {
          bad_page = 1;
          return;
        }
        for (int c = lane; c < kb / 16; c += 32) cp_async16(ks + pg * kb + 16 * c, kg + 16 * c);
        for (int c = lane; c < vb / 16; c += 32) cp_async16(vs + pg * vb + 16 * c, vg + 16 * c);
      }
      return;
    }
    const uint8_t* kg = main_row(lo, a.cp, 0, layer, seq, h, t0, &bad);
    const uint8_t* vg = main_row(lo, a.cp, 1, layer, seq, h, t0, &bad);
    for (int c = lane; c < C::KSTAGE / 16; c += 32) cp_async16(ks + 16 * c, kg + 16 * c);
    for (int c = lane; c < C::VSTAGE / 16; c += 32) cp_async16(vs + 16 * c, vg + 16 * c);
  };

  // ---- per-warp pipeline over this CTA's groups --------------------------------
  const int first = tb + warp;
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    issue(first + kWarps * i, i);
    cp_async_commit();
  }
  for (int it = 0;; ++it) {
    const int tile = first + kWarps * it;
    if (tile >= te) break;
    issue(tile + kWarps * (kStages - 1), (it + kStages - 1) % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();

    float S[2][NT][4];
#pragma unroll
    for (int mu = 0; mu < 2; ++mu)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) S[mu][nt][0] = S[mu][nt][1] = S[mu][nt][2] = S[mu][nt][3] = 0.f;
    float p[NT][4];

    if (tile < n_m) {
      // ---------------- packed group from shared memory ----------------
      const int t0 = tile * kTile;
      const int n_valid = min(kTile, qe - t0);
      const uint8_t* ksm = wst + (it % kStages) * C::STAGE;
      const uint8_t* vsm = ksm + C::VOFF;
      if constexpr (C::KCH) {
        // per-channel K: block c = channel c over the group's 32 tokens; the
        // channel scales multiply the query columns
#pragma unroll
        for (int kc = 0; kc < C::KC; ++kc) {
          const int c = 32 * (kc >> 1) + 8 * tq + 2 * (kc & 1);
          const uint8_t* b1p = ksm + c * C::KBB;
          const uint8_t* b2p = b1p + 4 * C::KBB;
          const uint8_t* b3p = b1p + C::KBB;
          const uint8_t* b4p = b1p + 5 * C::KBB;
          const uint32_t x12 = ld_u16(b1p + 2 + 2 * gq) | (ld_u16(b2p + 2 + 2 * gq) << 16);
          const uint32_t x34 = ld_u16(b3p + 2 + 2 * gq) | (ld_u16(b4p + 2 + 2 * gq) << 16);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float4 v = qsm[(kc * NT + nt) * 32 + lane];
            const uint32_t bq0 = pack_h2(split_part(v.x * block_scale(b1p), lo_part),
                                         split_part(v.y * block_scale(b2p), lo_part));
            const uint32_t bq1 = pack_h2(split_part(v.z * block_scale(b3p), lo_part),
                                         split_part(v.w * block_scale(b4p), lo_part));
#pragma unroll
            for (int mu = 0; mu < 2; ++mu)
              mma16816(S[mu][nt], code_pair<4>(x12, 2 * mu), code_pair<4>(x12, 2 * mu + 1),
                       code_pair<4>(x34, 2 * mu), code_pair<4>(x34, 2 * mu + 1), bq0, bq1);
          }
        }
      } else {
        // per-token K: each K block's scale multiplies its partial scores
#pragma unroll
        for (int kb = 0; kb < D / C::KG; ++kb) {
          float acc[2][NT][4];
#pragma unroll
          for (int mu = 0; mu < 2; ++mu)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[mu][nt][0] = acc[mu][nt][1] = acc[mu][nt][2] = acc[mu][nt][3] = 0.f;
#pragma unroll
          for (int ss = 0; ss < C::KSPB; ++ss) {
            const int s = kb * C::KSPB + ss;
#pragma unroll
            for (int mu = 0; mu < 2; ++mu) {
              const int ra = 4 * gq + 2 * mu;
              uint32_t wa[4], wb[4];
              k_token_pairs<C>(ksm + ra * C::KROW + kb * C::KBB + 2 + ss * C::KSPAN, tq, wa);
              k_token_pairs<C>(ksm + (ra + 1) * C::KROW + kb * C::KBB + 2 + ss * C::KSPAN, tq, wb);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                uint32_t b0, b1;
                qfrag(2 * s, nt, b0, b1);
                mma16816(acc[mu][nt], wa[0], wb[0], wa[1], wb[1], b0, b1);
                qfrag(2 * s + 1, nt, b0, b1);
                mma16816(acc[mu][nt], wa[2], wb[2], wa[3], wb[3], b0, b1);
              }
            }
          }
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            const float sa = block_scale(ksm + (4 * gq + 2 * mu) * C::KROW + kb * C::KBB);
            const float sb = block_scale(ksm + (4 * gq + 2 * mu + 1) * C::KROW + kb * C::KBB);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              S[mu][nt][0] += acc[mu][nt][0] * sa;
              S[mu][nt][1] += acc[mu][nt][1] * sa;
              S[mu][nt][2] += acc[mu][nt][2] * sb;
              S[mu][nt][3] += acc[mu][nt][3] * sb;
            }
          }
        }
      }
      online_softmax<C>(ws, S, n_valid, gq, qscale, p);
      // V: P^T per V block, O^T += V^T P^T
#pragma unroll
      for (int bv = 0; bv < D / C::VG; ++bv) {
        uint32_t pb[2][NT][2];
#pragma unroll
        for (int mu = 0; mu < 2; ++mu) {
          const int ra = 4 * gq + 2 * mu;
          const float sva = block_scale(vsm + ra * C::VROW + bv * C::VBB);
          const float svb = block_scale(vsm + (ra + 1) * C::VROW + bv * C::VBB);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float pa = ra < n_valid ? p[nt][2 * mu] * sva : 0.f;
            const float pbb = ra + 1 < n_valid ? p[nt][2 * mu + 1] * svb : 0.f;
            p_fragments(pa, pbb, pb[mu][nt][0], pb[mu][nt][1]);
          }
        }
#pragma unroll
        for (int ss = 0; ss < C::VSPB; ++ss) {
          const int s = bv * C::VSPB + ss;
          const int off = bv * C::VBB + 2 + ss * C::VSPAN;
#pragma unroll
          for (int mu = 0; mu < 2; ++mu) {
            const int T1 = 8 * tq + 2 * mu;
            uint32_t x12[4], x34[4];
            v_pair4<C>(vsm + T1 * C::VROW + off, vsm + (T1 + 4) * C::VROW + off, gq, x12);
            v_pair4<C>(vsm + (T1 + 1) * C::VROW + off, vsm + (T1 + 5) * C::VROW + off, gq, x34);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma16816(ws.o[2 * s][nt], x12[0], x12[1], x34[0], x34[1], pb[mu][nt][0], pb[mu][nt][1]);
              mma16816(ws.o[2 * s + 1][nt], x12[2], x12[3], x34[2], x34[3], pb[mu][nt][0], pb[mu][nt][1]);
            }
          }
        }
      }
    } else {
      // ---------------- 16-bit window group from global memory ----------------
      const int t0 = qe + (tile - n_m) * kTile;
      const int n_valid = min(kTile, T - t0);
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
            uint32_t q0, q1;
            qfrag(2 * s, nt, q0, q1);
            mma16816(S[mu][nt], a0, b0, a1, b1, q0, q1);
            qfrag(2 * s + 1, nt, q0, q1);
            mma16816(S[mu][nt], a2, b2, a3, b3, q0, q1);
          }
        }
      }
      online_softmax<C>(ws, S, n_valid, gq, qscale, p);
      uint32_t pb[2][NT][2];
#pragma unroll
      for (int mu = 0; mu < 2; ++mu) {
        const int ra = 4 * gq + 2 * mu;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          p_fragments(ra < n_valid ? p[nt][2 * mu] : 0.f, ra + 1 < n_valid ? p[nt][2 * mu + 1] : 0.f,
                      pb[mu][nt][0], pb[mu][nt][1]);
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
          }
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- merge the warps (shared memory), then the splits (workspace) -------------
  float* wm = reinterpret_cast<float*>(stage_base);  // [kWarps][g]
  float* wl = wm + kWarps * kMaxGqa;                  // [kWarps][g]
  float* wo = wl + kWarps * kMaxGqa;                  // [kWarps][g][D]
  float* obuf = wo + kWarps * kMaxGqa * D;            // [g][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float l = ws.l[nt];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    const int hh = 4 * nt + tq;
    if (hh < g) {
      if (gq == 0) {
        wm[warp * kMaxGqa + hh] = ws.m[nt];
        wl[warp * kMaxGqa + hh] = l;
      }
      float* orow = wo + (warp * kMaxGqa + hh) * D;
#pragma unroll
      for (int s = 0; s < C::NS; ++s)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ch = 32 * s + 4 * gq + 2 * e;
          orow[ch] = ws.o[2 * s + e][nt][0] + ws.o[2 * s + e][nt][1];
          orow[ch + 1] = ws.o[2 * s + e][nt][2] + ws.o[2 * s + e][nt][3];
        }
    }
  }
  __syncthreads();
  if (tid == 0 && bad_page) atomicOr(a.status, KVQ_DEV_PAGE);
  // CTA partial per head: M = max_w m_w, L = sum_w 2^(m_w - M) l_w, O likewise
  const int64_t unit = ((int64_t)li * lo.B + seq) * lo.H + h;
  float* part = a.partials + (unit * a.splits + split) * (int64_t)g * (D + 2);
  for (int e = tid; e < g * D; e += kThreadsMma) {
    const int hh = e / D, d = e % D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kMaxGqa + hh]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        const float sc = exp2f(wm[w * kMaxGqa + hh] - M);
        L += sc * wl[w * kMaxGqa + hh];
        O += sc * wo[(w * kMaxGqa + hh) * D + d];
      }
    }
    if (a.splits == 1) {
      obuf[e] = L > 0.f ? O / L : 0.f;
    } else {
      part[hh * (D + 2) + 2 + d] = O;
      if (d == 0) {
        part[hh * (D + 2)] = M;
        part[hh * (D + 2) + 1] = L;
      }
    }
  }
  if (a.splits > 1) {
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(a.tickets + unit, 1u) == (unsigned)(a.splits - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const float* base = a.partials + unit * a.splits * (int64_t)g * (D + 2);
    for (int e = tid; e < g * D; e += kThreadsMma) {
      const int hh = e / D, d = e % D;
      float M = -INFINITY;
      for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, __ldcg(base + ((int64_t)sp * g + hh) * (D + 2)));
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int sp = 0; sp < a.splits; ++sp) {
          const float* pp = base + ((int64_t)sp * g + hh) * (D + 2);
          const float w = exp2f(__ldcg(pp) - M);
          L += w * __ldcg(pp + 1);
          O += w * __ldcg(pp + 2 + d);
        }
      }
      obuf[e] = L > 0.f ? O / L : 0.f;
    }
    if (tid == 0) a.tickets[unit] = 0;
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

template <class C>
cudaError_t launch_mma(const DecodeArgs& a, cudaStream_t st) {
  static_assert(C::SMEM >= C::QSM + (2 * kWarps * kMaxGqa + kWarps * kMaxGqa * C::D + kMaxGqa * C::D) * 4,
                "merge scratch must fit in the stage buffers");
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(a.splits, a.lo.H, a.n_layers * a.lo.B);
  decode_mma_kernel<C><<<grid, kThreadsMma, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

bool fmt_is(const FmtInfo& f, int bits, int group, int axis) {
  return f.bits == bits && f.group == group && f.axis == axis;
}

}  // namespace

// Tensor-core path when the cache fits it, else the generic path.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  const Layout& lo = a.lo;
  bool ok = !lo.tiered && !(lo.flags & KVQ_K_PRE_ROPE);
  if (lo.ring) ok = ok && lo.dtype == KVQ_DT_F16 && !(lo.flags & (KVQ_ROTATE_K | KVQ_ROTATE_V));
  if (lo.paged) ok = ok && (lo.pt == 16 || lo.pt == 32);
  if (ok) {
    const FmtInfo &k = lo.kf, &v = lo.vf;
    const int T = KVQ_AXIS_TOKEN, CH = KVQ_AXIS_CHANNEL;
    if (lo.D == 128 && lo.g <= 4) {
      if (fmt_is(k, 4, 32, CH) && fmt_is(v, 4, 32, T)) return launch_mma<Cfg<128, 1, KF_CH4, 32, VF_T4, 32>>(a, st);
      if (fmt_is(k, 4, 128, T) && fmt_is(v, 4, 128, T)) return launch_mma<Cfg<128, 1, KF_T4, 128, VF_T4, 128>>(a, st);
      if (fmt_is(k, 4, 32, T) && fmt_is(v, 4, 32, T)) return launch_mma<Cfg<128, 1, KF_T4, 32, VF_T4, 32>>(a, st);
      if (fmt_is(k, 8, 32, T) && fmt_is(v, 8, 32, T)) return launch_mma<Cfg<128, 1, KF_T8, 32, VF_T8, 32>>(a, st);
    }
    if (lo.D == 256 && lo.g <= 8) {
      if (fmt_is(k, 4, 128, T) && fmt_is(v, 4, 128, T)) return launch_mma<Cfg<256, 2, KF_T4, 128, VF_T4, 128>>(a, st);
      if (fmt_is(k, 3, 128, T) && fmt_is(v, 3, 128, T)) return launch_mma<Cfg<256, 2, KF_T3, 128, VF_T3, 128>>(a, st);
    }
  }
  return launch_decode_generic(a, st);
}

}  // namespace kvq
