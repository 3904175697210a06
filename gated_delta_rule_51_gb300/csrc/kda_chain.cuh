// kda_chain.cuh -- the fused chunked KDA forward kernel for sm_103a (a template; kda_chain.cu
// instantiates the usual variants, kda_chain_precise.cu the precise-state ones).
//
// One CTA walks one run of 16-token chunks of one (sequence, head) -- a whole
// sequence, or one segment of a long one -- and keeps the 128 x 128 fp32 state
// on chip for the whole run (FlashKDA works in chunks of 16 tokens and updates the
// state in fp32; instagit index, kernel articles).  Per chunk, with S the state on entry:
//
//   G    = within-chunk inclusive cumsum of the base-2 log-decay (per channel)
//   Akk  = tril(beta_i * (kh*2^G)(kh*2^-G)^T, -1)   Aqk = tril((qh*2^G)(kh*2^-G)^T, 0)
//          (the Gram factors are taken about a = G_C / 2, 2^(G-a) and 2^(a-G), so that
//          no factor leaves 2^+-125 while |G_C| <= 250; beyond that the chunk sets the
//          gate-range error bit)
//   Tm   = (I + Akk)^-1 Diag(beta)          (forward substitution, fp32)
//   W    = Tm (kh*2^G),  U = Tm v,  Vn = U - W S
//   O    = scale * ((qh*2^G) S + Aqk Vn)
//   S'   = Diag(2^G_C) S + (kh*2^(G_C-G))^T Vn
//
// Warp roles (256 threads, two CTAs per SM):
//   warps 0-3   prologue, two pairs (even / odd chunks); a pair splits the 128
//               channels: gate, cumsum, L2 norms, Gram matrices (tf32 warp MMA),
//               inverse, W (bf16 warp MMA).  The tcgen05 operands are written in
//               place over the tiles they are made from: q -> qh*2^G, k -> kfac
//               (hi), g -> kfac (lo), and a bf16 copy of kh*2^G next to q, which
//               the W product then overwrites with -W.
//   warps 4-7   epilogue, one TMEM lane quarter each: Vn read-out (split into
//               bf16 hi + lo), outputs, state decay + bf16 copy of S^T for the
//               next chunk's A operand.  Lane 0 of warp 4 issues every tcgen05
//               MMA; lane 0 of warp 5 issues the TMA loads of each stage of a
//               four-stage ring.
// State GEMMs in the M = V = 128 orientation:
//               D1 = V^T Tm^T + S^T [-W^T | (qh 2^G)^T]   (N = 32)
//               D2 += Vn^T kfac ;  D1[:,16:] += Vn^T Aqk^T
// TMEM (256 columns): [0,128) S^T fp32 accumulator, [128,192) S^T as packed
// bf16 (A operand read straight from TMEM), [192,256) two 32-column D1 tiles.
//
// Precision: the S-side GEMM runs on bf16 copies of S^T, W and qh*2^G; the
// rank-16 state update, U and Aqk*Vn use a split-bf16 (hi + lo) scheme, and
// the Grams use tf32.  With a gate that decays, the rounding of the bf16 copies
// fades within a few chunks; with one that hardly decays it builds up (about
// 1.9e-3 rel-Fro on the fp32 state at lower_bound 0), so the precise-state
// variant (kChainPrecise) also splits S^T, W and the kh*2^G tile W is made from
// into bf16 hi + lo (320 TMEM columns, 4 KB more per stage: one CTA per SM).
#pragma once
#include <atomic>
#include <type_traits>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

// Eight warps, two CTAs per SM: sixteen warps per SM leave 128 registers a thread.
constexpr int kThreads = 256;
constexpr int kStages = 4;
constexpr int kWarpProlog0 = 0;       // prologue warps 0-3: two pairs, one pair per chunk
constexpr int kWarpEpi0 = 4;          // epilogue warps 4-7; lane 0 of warp 4 issues the MMAs
constexpr int kWarpTma = 5;           // lane 0 of epilogue warp 5 issues the TMA loads
constexpr uint32_t kBarEpi = 3;       // named barrier of the epilogue warps
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemColsPrecise = 512;   // precise-state runs: 320 columns used
constexpr uint32_t kColSlo = 256;            // precise-state runs: the bf16 remainder of S^T
constexpr uint32_t kColState = 0;
constexpr uint32_t kColSbf = 128;
constexpr uint32_t kColD1 = 192;
constexpr float kLog2e = 1.4426950408889634f;

// One chunk's stage.  Offsets of the 128-byte swizzled regions are multiples
// of 1024 bytes.  X block b (b = 0, 1 for channels 64b .. 64b+63) is the K-major
// B operand of the S-side GEMM: rows 0-15 = -W (first holds bf16 kh*2^G),
// rows 16-31 = qh*2^G (first holds the q tile, as the TMA box lands there).
struct Stage {
  uint8_t X[2][4096];
  uint8_t K[4096];        // k tile -> kfac hi   (MN-major B of the state update)
  uint8_t G[4096];        // g tile -> kfac lo
  uint8_t V[4096];        // v tile (MN-major A of U^T = V^T Tm^T)
};
static_assert(sizeof(Stage) == 20480, "stage size (multiple of 1024 for the swizzled regions)");
// Precise-state stage: block b of WL holds the bf16 remainder of kh*2^G, then of -W (16 rows,
// laid out as rows 0-15 of X[b]); it is a second K-major B operand of the S-side GEMM.
struct StagePrecise : Stage {
  uint8_t WL[2][2048];
};
static_assert(sizeof(StagePrecise) == 24576, "precise stage size (multiple of 1024)");
struct StageSmall {       // the unswizzled operands of the same chunk
  uint8_t TPhi[1024];     // [Tm ; 0] [32 rows][16] K-major, no swizzle
  uint8_t TPlo[1024];
  uint8_t AQhi[512];      // Aqk [16][16] K-major, no swizzle
  uint8_t AQlo[512];
  float gamC[128];        // 2^G_C per channel
};
static_assert(sizeof(StageSmall) == 3584, "small stage size");
struct PairScratch {      // exchange area of one prologue pair (fp32, token indices)
  float normx[2][16][2];  // per-warp partial |q|^2, |k|^2
  float GkX[16][16];      // warp 1's partial Gk, then -beta_i Gk[i][m] stored at [m][i]
  float Gq0[16][16];      // warp 0's partial Gq
  int okf[2][2];          // both warps' wait results, by iteration parity
};
template <bool kPrecise>
struct SmemLayoutT {
  typename std::conditional<kPrecise, StagePrecise, Stage>::type st[kStages];
  StageSmall sm[kStages];
  uint8_t vn_hi[4096];    // Vn^T [128 v][16 tok] K-major, no swizzle
  uint8_t vn_lo[4096];
  uint8_t ostage[16][256];  // one chunk's bf16 outputs [token][v], for coalesced stores
  PairScratch ps[2];
};
template <bool kPrecise>
constexpr size_t chain_smem_bytes_t() { return sizeof(SmemLayoutT<kPrecise>) + 1024; }

// byte offset of the 16-byte chunk holding channels [8 j16', 8 j16' + 8) of row r
// in a [16 x 64] bf16 tile with the 128-byte swizzle (j16 = chunk index 0..7)
__device__ __forceinline__ uint32_t sw_off(int r, int j16) {
  return (uint32_t)(r * 128 + ((j16 ^ (r & 7)) << 4));
}
// byte offset of (row n, k) in a K-major, unswizzled operand with 16 k per row:
// 8x16-byte core matrices, LBO = 128 (k direction), SBO = 256 (row direction)
__device__ __forceinline__ uint32_t ns_off(int n, int k) {
  return (uint32_t)((n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// split x into hi + lo bf16 parts (hi = RNE(x), lo = RNE(x - hi))
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  float r = x - __bfloat162float(h);
  __nv_bfloat16 l = __float2bfloat16_rn(r);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}
// split two floats into packed hi and lo bf16x2 words
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo_to_f32(hi), b - bf16hi_to_f32(hi));
}
// packed fp32x2 arithmetic on pairs of floats
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ void fmul2(float& a0, float& a1, float b0, float b1) {
  uint64_t c;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(f2pack(a0, a1)), "l"(f2pack(b0, b1)));
  f2unpack(c, a0, a1);
}
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2pack(a0, a1)), "l"(f2pack(b0, b1)), "l"(f2pack(c0, c1)));
  f2unpack(r, d0, d1);
}
__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  uint64_t c;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(f2pack(a0, a1)), "l"(f2pack(b0, b1)));
  f2unpack(c, a0, a1);
}
// (a0, a1) * (b0, b1) with one packed fp32x2 multiply
__device__ __forceinline__ void mul2(uint32_t& x0, uint32_t& x1, float b0, float b1) {
  uint64_t a, b, c;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "r"(x0), "r"(x1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(c) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=r"(x0), "=r"(x1) : "l"(c));
}

// Column group j (32 bf16 values, 16 packed words) of row `row` of a stored 128 x 128 state copy.
// The copy is kept piece-major: 16-byte piece q (columns 8 q .. 8 q + 7) of row r at piece
// index q * 128 + r, so that the 32 lanes of a warp (consecutive rows) write 512 contiguous bytes.
__device__ __forceinline__ void store_packed16(uint16_t* copy, int row, int j, const uint32_t (&pk)[16]) {
  uint4* d = reinterpret_cast<uint4*>(copy);
#pragma unroll
  for (int t = 0; t < 4; ++t)
    d[(4 * j + t) * 128 + row] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
}

// Column group j of a stored copy (as store_packed16) plus 32 fp32 values, rounded to bf16 again:
// a correction run's part added to what its segment's run stored.
__device__ __forceinline__ void add_to_copy(uint16_t* copy, int row, int j, const float (&x)[32]) {
  uint4* d = reinterpret_cast<uint4*>(copy);
  uint4 w[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) w[t] = d[(4 * j + t) * 128 + row];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t a[4] = {w[t].x, w[t].y, w[t].z, w[t].w};
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      o[u] = pack_bf16x2(bf16lo_to_f32(a[u]) + x[8 * t + 2 * u], bf16hi_to_f32(a[u]) + x[8 * t + 2 * u + 1]);
    d[(4 * j + t) * 128 + row] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Named barrier of one prologue pair (64 threads; ids 1 and 2).
__device__ __forceinline__ void pair_bar(int pair) { named_bar(1 + pair, 64); }

// Prepare the tcgen05 operands of one chunk with a pair of warps; warp w of the
// pair handles channels [64 w, 64 w + 64) (passes p = 2 w, 2 w + 1 of 32 channels).
// Lane (gid, tig) holds tokens ra = 2 gid and rb = 2 gid + 1 and, in pass p,
// channels 32 p + 8 tig + j (j < 8).  For the Gram warp MMAs the physical tokens
// 2 gid / 2 gid + 1 play the fragment rows gid / gid + 8, and the channel pair
// (8 tig + 2 s, + 1) the k positions (tig, tig + 4) of k-step s; the partial
// Grams of the two warps are summed through shared memory.
// A reverse run of the backward (kBwd, rev) scales qh*2^G by qscale and writes Aqk transposed
// and scaled: the B operands of its update (dO^T scale Q_p) and of its S-side GEMM (dO^T scale P).
template <int kFlags, bool kPrecise, bool kBwd>
__device__ __forceinline__ void prologue_pair_chunk(Stage& st, uint8_t* wl, StageSmall& sm, PairScratch& sc, int pair,
                                                    int w, int nv,
                                                    int* err, const float nr, const float lbl2,
                                                    const float* __restrict__ dtb, float beta_a, float beta_b,
                                                    int lane, bool v_used, bool rev, float qscale) {
  constexpr bool gate_pre = kFlags & kGatePreactivated;
  constexpr bool gate_sp = kFlags & kGateSoftplus;   // then nr = log2(e), lbl2 = -exp(A_log)
  // the safe gate keeps |G_C| <= 16 * 5 * log2(e) < 126, where the Gram factors 2^+-G are
  // exact as they are; the other two gates factor about the anchor a = G_C / 2
  constexpr bool anchored = gate_pre || gate_sp;
  const int gid = lane >> 2, tig = lane & 3;
  const int ra = 2 * gid, rb = 2 * gid + 1;
  const bool va = ra < nv, vb = rb < nv;
  const bool partial = nv < kChunk;

  // ---- L2 norms of q and k: partial sums over this warp's 64 channels
  {
    float sq[2] = {0.f, 0.f}, sk[2] = {0.f, 0.f};
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const int p = 2 * w + pp;
      const int j16 = 4 * (p & 1) + tig;
      const uint8_t* qb = st.X[p >> 1] + 2048;
      const uint8_t* kb = st.K + 2048 * (p >> 1);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = ra + hr;
        const uint4 wq = *reinterpret_cast<const uint4*>(qb + sw_off(r, j16));
        const uint4 wk = *reinterpret_cast<const uint4*>(kb + sw_off(r, j16));
        const uint32_t aq[4] = {wq.x, wq.y, wq.z, wq.w}, ak[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float q0 = bf16lo_to_f32(aq[u]), q1 = bf16hi_to_f32(aq[u]);
          const float k0 = bf16lo_to_f32(ak[u]), k1 = bf16hi_to_f32(ak[u]);
          sq[hr] = fmaf(q0, q0, fmaf(q1, q1, sq[hr]));
          sk[hr] = fmaf(k0, k0, fmaf(k1, k1, sk[hr]));
        }
      }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        sq[hr] += __shfl_xor_sync(0xffffffffu, sq[hr], m);
        sk[hr] += __shfl_xor_sync(0xffffffffu, sk[hr], m);
      }
    }
    if (tig == 0) {
      *reinterpret_cast<float2*>(&sc.normx[w][ra][0]) = make_float2(sq[0], sk[0]);
      *reinterpret_cast<float2*>(&sc.normx[w][rb][0]) = make_float2(sq[1], sk[1]);
    }
  }
  pair_bar(pair);
  float rq[2], rk[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const float2 a = *reinterpret_cast<const float2*>(&sc.normx[0][ra + hr][0]);
    const float2 b = *reinterpret_cast<const float2*>(&sc.normx[1][ra + hr][0]);
    const bool valid = hr == 0 ? va : vb;
    constexpr bool norm = !(kFlags & kNoQkL2Norm);
    rq[hr] = valid ? (norm ? rsqrt_approx(a.x + b.x + 1e-6f) : 1.f) : 0.f;
    rk[hr] = valid ? (norm ? rsqrt_approx(a.y + b.y + 1e-6f) : 1.f) : 0.f;
  }

  float ck0[4] = {0, 0, 0, 0}, ck1[4] = {0, 0, 0, 0}, cq0[4] = {0, 0, 0, 0}, cq1[4] = {0, 0, 0, 0};
#pragma unroll 1
  for (int pp = 0; pp < 2; ++pp) {
    const int p = 2 * w + pp;
    const int j16 = 4 * (p & 1) + tig;
    const int ch0 = 32 * p + 8 * tig;
    float nrdb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (!gate_pre) {
      const float4 d0 = *reinterpret_cast<const float4*>(dtb + ch0);
      const float4 d1 = *reinterpret_cast<const float4*>(dtb + ch0 + 4);
      nrdb[0] = nr * d0.x; nrdb[1] = nr * d0.y; nrdb[2] = nr * d0.z; nrdb[3] = nr * d0.w;
      nrdb[4] = nr * d1.x; nrdb[5] = nr * d1.y; nrdb[6] = nr * d1.z; nrdb[7] = nr * d1.w;
    }
    uint8_t* qb = st.X[p >> 1] + 2048;
    uint8_t* wb = st.X[p >> 1];
    uint8_t* kb = st.K + 2048 * (p >> 1);
    uint8_t* gb = st.G + 2048 * (p >> 1);
    float q[2][8], k[2][8], G[2][8];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = ra + hr;
      const bool valid = hr == 0 ? va : vb;
      uint4 wq = *reinterpret_cast<const uint4*>(qb + sw_off(r, j16));
      uint4 wk = *reinterpret_cast<const uint4*>(kb + sw_off(r, j16));
      const uint4 wg = *reinterpret_cast<const uint4*>(gb + sw_off(r, j16));
      if (partial && !valid) {
        wq = make_uint4(0u, 0u, 0u, 0u);
        wk = make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t aq[4] = {wq.x, wq.y, wq.z, wq.w}, ak[4] = {wk.x, wk.y, wk.z, wk.w};
      const uint32_t ag[4] = {wg.x, wg.y, wg.z, wg.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        q[hr][2 * u] = bf16lo_to_f32(aq[u]);
        q[hr][2 * u + 1] = bf16hi_to_f32(aq[u]);
        k[hr][2 * u] = bf16lo_to_f32(ak[u]);
        k[hr][2 * u + 1] = bf16hi_to_f32(ak[u]);
        // gate: base-2 log-decay lb * log2(e) * sigmoid(exp(A_log) (g + dt_bias)), or
        // -exp(A_log) log2(1 + 2^y) with y = log2(e) (g + dt_bias) (the gate without a
        // lower bound: log2(e) softplus), or log2(e) g for a gate activated by the
        // caller; 0 past the end
        float r0, r1;
        if (gate_pre) {
          r0 = bf16lo_to_f32(ag[u]);
          r1 = bf16hi_to_f32(ag[u]);
          const float lv = valid ? kLog2e : 0.f;
          fmul2(r0, r1, lv, lv);
        } else if (gate_sp) {
          float y0, y1;
          ffma2(y0, y1, nr, nr, bf16lo_to_f32(ag[u]), bf16hi_to_f32(ag[u]), nrdb[2 * u], nrdb[2 * u + 1]);
          // log2(1 + 2^y) = max(y, 0) + log2(1 + 2^-|y|)
          float t0 = ex2_approx(-fabsf(y0)), t1 = ex2_approx(-fabsf(y1));
          fadd2(t0, t1, 1.f, 1.f);
          r0 = fmaxf(y0, 0.f) + lg2_approx(t0);
          r1 = fmaxf(y1, 0.f) + lg2_approx(t1);
          const float lv = valid ? lbl2 : 0.f;
          fmul2(r0, r1, lv, lv);
        } else {
          float x0, x1;
          ffma2(x0, x1, nr, nr, bf16lo_to_f32(ag[u]), bf16hi_to_f32(ag[u]), nrdb[2 * u], nrdb[2 * u + 1]);
          float t0 = ex2_approx(x0), t1 = ex2_approx(x1);
          fadd2(t0, t1, 1.f, 1.f);
          r0 = rcp_approx(t0);
          r1 = rcp_approx(t1);
          const float lv = valid ? lbl2 : 0.f;
          fmul2(r0, r1, lv, lv);
        }
        // (a token decaying by 2^-1000 or more wipes every factor that spans it to an fp32
        // zero: clamping its log-decay there changes no result and keeps sums finite)
        if (anchored) {
          r0 = fmaxf(r0, -1000.f);
          r1 = fmaxf(r1, -1000.f);
        }
        G[hr][2 * u] = (partial && !valid) ? 0.f : r0;
        G[hr][2 * u + 1] = (partial && !valid) ? 0.f : r1;
      }
    }
    // ---- within-chunk inclusive cumsum over tokens (pairs in a lane, scan over gid)
    float gC[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float pr = G[0][j] + G[1][j];
      float incl = pr;
#pragma unroll
      for (int d = 1; d <= 4; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, 4 * d);
        if (gid >= d) incl += y;
      }
      const float excl = incl - pr;
      G[0][j] = excl + G[0][j];
      G[1][j] = incl;
      gC[j] = __shfl_sync(0xffffffffu, incl, 28 + tig);
    }
    // The anchored factors stay finite while the chunk decays by at most 2^-250 on every
    // channel.  Past that the precise-state kernels (the ones these gates run) take the
    // direct route below; the others flag the chunk.
    if (anchored) {
      bool bad = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) bad = bad || !(fabsf(gC[j]) <= 250.f);
      const bool out_of_range = __any_sync(0xffffffffu, bad);
      if constexpr (!kPrecise) {
        if (out_of_range && lane == 0) atomicOr(err, kErrGateRange);
      } else if (out_of_range) {
        // ---- direct route for this pass's 32 channels: every factor is a power of two of a
        //      non-positive exponent (2^G, 2^(G_C - G), and 2^(G_i - G_j) per pair j <= i), so
        //      nothing overflows and what underflows is below fp32's reach in the result too
        float kh[2][8], qh[2][8];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            kh[hr][j] = k[hr][j] * rk[hr];
            qh[hr][j] = q[hr][j] * rq[hr];
          }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const uint32_t o = sw_off(ra + hr, j16);
          uint32_t qw[4], kw[4], kl[4], hw[4], lw[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j0 = 2 * u, j1 = 2 * u + 1;
            const float e0 = ex2_approx(G[hr][j0]), e1 = ex2_approx(G[hr][j1]);
            const float f0 = ex2_approx(gC[j0] - G[hr][j0]), f1 = ex2_approx(gC[j1] - G[hr][j1]);
            qw[u] = pack_bf16x2(qh[hr][j0] * e0, qh[hr][j1] * e1);
            split_bf16x2(kh[hr][j0] * e0, kh[hr][j1] * e1, kw[u], kl[u]);
            split_bf16x2(kh[hr][j0] * f0, kh[hr][j1] * f1, hw[u], lw[u]);
          }
          *reinterpret_cast<uint4*>(qb + o) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
          *reinterpret_cast<uint4*>(wb + o) = make_uint4(kw[0], kw[1], kw[2], kw[3]);
          *reinterpret_cast<uint4*>(wl + 2048 * (p >> 1) + o) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
          *reinterpret_cast<uint4*>(kb + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(gb + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        if (gid == 0) {
          float e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) e[j] = ex2_approx(gC[j]);
          *reinterpret_cast<float4*>(&sm.gamC[ch0]) = make_float4(e[0], e[1], e[2], e[3]);
          *reinterpret_cast<float4*>(&sm.gamC[ch0 + 4]) = make_float4(e[4], e[5], e[6], e[7]);
        }
        // Gram partials over the lane's 8 channels: token jt's values come from lane
        // (gid = jt / 2, same tig), then the 4 lanes of a tig group are summed
        float pk[2][16], pq[2][16];
#pragma unroll
        for (int jt = 0; jt < 16; ++jt) {
          const int src = 4 * (jt >> 1) + tig;
          float Gj[8], kj[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            Gj[c] = __shfl_sync(0xffffffffu, G[jt & 1][c], src);
            kj[c] = __shfl_sync(0xffffffffu, kh[jt & 1][c], src);
          }
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float sk = 0.f, sq = 0.f;
            if (jt <= ra + hr) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const float e = ex2_approx(G[hr][c] - Gj[c]) * kj[c];
                sk = fmaf(kh[hr][c], e, sk);
                sq = fmaf(qh[hr][c], e, sq);
              }
            }
            pk[hr][jt] = sk;
            pq[hr][jt] = sq;
          }
        }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
          for (int jt = 0; jt < 16; ++jt)
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {
              pk[hr][jt] += __shfl_xor_sync(0xffffffffu, pk[hr][jt], m);
              pq[hr][jt] += __shfl_xor_sync(0xffffffffu, pq[hr][jt], m);
            }
        // into the fragment accumulators: rows ra (c[0], c[1]) and rb (c[2], c[3]); token
        // columns 4 tig, 4 tig + 2 in ck0 / cq0 and 4 tig + 1, 4 tig + 3 in ck1 / cq1
#pragma unroll
        for (int jt = 0; jt < 16; ++jt) {
          if (jt == 4 * tig) {
            ck0[0] += pk[0][jt]; ck0[2] += pk[1][jt]; cq0[0] += pq[0][jt]; cq0[2] += pq[1][jt];
          } else if (jt == 4 * tig + 2) {
            ck0[1] += pk[0][jt]; ck0[3] += pk[1][jt]; cq0[1] += pq[0][jt]; cq0[3] += pq[1][jt];
          } else if (jt == 4 * tig + 1) {
            ck1[0] += pk[0][jt]; ck1[2] += pk[1][jt]; cq1[0] += pq[0][jt]; cq1[2] += pq[1][jt];
          } else if (jt == 4 * tig + 3) {
            ck1[1] += pk[0][jt]; ck1[3] += pk[1][jt]; cq1[1] += pq[0][jt]; cq1[3] += pq[1][jt];
          }
        }
        continue;
      }
    }
    float eA[8];   // 2^a with the anchor a = G_C / 2 (anchored), else 2^G_C
#pragma unroll
    for (int j = 0; j < 8; ++j) eA[j] = ex2_approx(anchored ? 0.5f * gC[j] : gC[j]);
    // ---- decay-scaled operands: the Gram factors about the anchor (2^(G-a), 2^(a-G))
    float kg[2][8], ki[2][8], qg[2][8];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float d0 = anchored ? fmaf(-0.5f, gC[j], G[hr][j]) : G[hr][j];
        const float d1 = anchored ? fmaf(-0.5f, gC[j + 1], G[hr][j + 1]) : G[hr][j + 1];
        const float gam0 = ex2_approx(d0), gam1 = ex2_approx(d1);
        const float gin0 = ex2_approx(-d0), gin1 = ex2_approx(-d1);
        float kh0 = k[hr][j], kh1 = k[hr][j + 1];
        fmul2(kh0, kh1, rk[hr], rk[hr]);
        float qh0 = q[hr][j], qh1 = q[hr][j + 1];
        fmul2(qh0, qh1, rq[hr], rq[hr]);
        kg[hr][j] = kh0; kg[hr][j + 1] = kh1;
        fmul2(kg[hr][j], kg[hr][j + 1], gam0, gam1);
        ki[hr][j] = kh0; ki[hr][j + 1] = kh1;
        fmul2(ki[hr][j], ki[hr][j + 1], gin0, gin1);
        qg[hr][j] = qh0; qg[hr][j + 1] = qh1;
        fmul2(qg[hr][j], qg[hr][j + 1], gam0, gam1);
      }
    // ---- Gram partials over this pass's 32 channels (tf32 warp MMA)
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      const int j = 2 * s2;
      // fp32 bit patterns; the tf32 MMA uses their top 19 bits
      const uint32_t ak[4] = {__float_as_uint(kg[0][j]), __float_as_uint(kg[1][j]), __float_as_uint(kg[0][j + 1]),
                              __float_as_uint(kg[1][j + 1])};
      const uint32_t aq[4] = {__float_as_uint(qg[0][j]), __float_as_uint(qg[1][j]), __float_as_uint(qg[0][j + 1]),
                              __float_as_uint(qg[1][j + 1])};
      const uint32_t b0[2] = {__float_as_uint(ki[0][j]), __float_as_uint(ki[0][j + 1])};
      const uint32_t b1[2] = {__float_as_uint(ki[1][j]), __float_as_uint(ki[1][j + 1])};
      mma_tf32_16x8x8(ck0, ak, b0);
      mma_tf32_16x8x8(ck1, ak, b1);
      mma_tf32_16x8x8(cq0, aq, b0);
      mma_tf32_16x8x8(cq1, aq, b1);
    }
    // ---- operand tiles, written in place: qh*2^G and kh*2^G (anchored: the factor times 2^a),
    //      kfac = kh*2^(G_C-G) (2^-G times 2^G_C; anchored: 2^(a-G) times 2^a)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const uint32_t o = sw_off(ra + hr, j16);
      {
        uint32_t qw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float a0 = qg[hr][2 * u], a1 = qg[hr][2 * u + 1];
          if (anchored) fmul2(a0, a1, eA[2 * u], eA[2 * u + 1]);
          if (kBwd && rev) fmul2(a0, a1, qscale, qscale);
          qw[u] = pack_bf16x2(a0, a1);
        }
        *reinterpret_cast<uint4*>(qb + o) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      }
      {
        uint32_t kw[4], kl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float b0 = kg[hr][2 * u], b1 = kg[hr][2 * u + 1];
          if (anchored) fmul2(b0, b1, eA[2 * u], eA[2 * u + 1]);
          if (kPrecise) split_bf16x2(b0, b1, kw[u], kl[u]);
          else kw[u] = pack_bf16x2(b0, b1);
        }
        *reinterpret_cast<uint4*>(wb + o) = make_uint4(kw[0], kw[1], kw[2], kw[3]);
        if (kPrecise) *reinterpret_cast<uint4*>(wl + 2048 * (p >> 1) + o) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f0 = ki[hr][2 * u], f1 = ki[hr][2 * u + 1];
        fmul2(f0, f1, eA[2 * u], eA[2 * u + 1]);
        split_bf16x2(f0, f1, hw[u], lw[u]);
      }
      *reinterpret_cast<uint4*>(kb + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(gb + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    if (gid == 0) {   // 2^G_C (anchored: (2^a)^2)
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = anchored ? eA[j] * eA[j] : eA[j];
      *reinterpret_cast<float4*>(&sm.gamC[ch0]) = make_float4(e[0], e[1], e[2], e[3]);
      *reinterpret_cast<float4*>(&sm.gamC[ch0 + 4]) = make_float4(e[4], e[5], e[6], e[7]);
    }
  }
  // ---- Gram exchange: warp 1 hands its Gk partial to warp 0, warp 0 its Gq partial
  //      to warp 1 (fragment row gid = token 2 gid, gid + 8 = 2 gid + 1; columns 2 tig,
  //      2 tig + 1, 8 + 2 tig, 9 + 2 tig = tokens 4 tig, 4 tig + 2, 4 tig + 1, 4 tig + 3)
  {
    float* dst = w == 0 ? &sc.Gq0[0][0] : &sc.GkX[0][0];
    const float* c0 = w == 0 ? cq0 : ck0;
    const float* c1 = w == 0 ? cq1 : ck1;
    *reinterpret_cast<float4*>(dst + ra * 16 + 4 * tig) = make_float4(c0[0], c1[0], c0[1], c1[1]);
    *reinterpret_cast<float4*>(dst + rb * 16 + 4 * tig) = make_float4(c0[2], c1[2], c0[3], c1[3]);
  }
  pair_bar(pair);
  // beta of the lane's tokens
  constexpr bool beta_pre = kFlags & kBetaPreactivated;
  const float sa = va ? (beta_pre ? beta_a : rcp_approx(1.f + ex2_approx(-beta_a * kLog2e))) : 0.f;
  const float sb = vb ? (beta_pre ? beta_b : rcp_approx(1.f + ex2_approx(-beta_b * kLog2e))) : 0.f;
  if (w == 0) {
    // full Gk = own partial + warp 1's; store column m of -Akk contiguous: AT[m][i] = -beta_i Gk[i][m]
    const float4 xa = *reinterpret_cast<const float4*>(&sc.GkX[ra][4 * tig]);
    const float4 xb = *reinterpret_cast<const float4*>(&sc.GkX[rb][4 * tig]);
    const float ka[4] = {ck0[0] + xa.x, ck1[0] + xa.y, ck0[1] + xa.z, ck1[1] + xa.w};
    const float kb[4] = {ck0[2] + xb.x, ck1[2] + xb.y, ck0[3] + xb.z, ck1[3] + xb.w};
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      sc.GkX[4 * tig + u][ra] = -sa * ka[u];
      sc.GkX[4 * tig + u][rb] = -sb * kb[u];
    }
    float bet[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) bet[i] = __shfl_sync(0xffffffffu, (i & 1) ? sb : sa, 4 * (i >> 1));
    __syncwarp();
    if (lane < 16) {
      // column j of X = (I + Akk)^-1 by forward substitution
      const int j = lane;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 15; ++m) {
        float a[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 t = *reinterpret_cast<const float4*>(&sc.GkX[m][4 * q4]);
          a[4 * q4] = t.x; a[4 * q4 + 1] = t.y; a[4 * q4 + 2] = t.z; a[4 * q4 + 3] = t.w;
        }
#pragma unroll
        for (int i = m + 1; i < 16; ++i) x[i] = fmaf(a[i], x[m], x[i]);
      }
      float bj = bet[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) bj = (j == i) ? bet[i] : bj;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint16_t hi, lo;
        split_bf16(x[i] * bj, hi, lo);
        const uint32_t o = ns_off(i, j);
        *reinterpret_cast<uint16_t*>(sm.TPhi + o) = hi;
        *reinterpret_cast<uint16_t*>(sm.TPlo + o) = lo;
      }
    }
  } else {
    // Aqk = own Gq partial + warp 0's, inclusive lower triangle, split bf16 (4 tokens per store)
    const float4 xa = *reinterpret_cast<const float4*>(&sc.Gq0[ra][4 * tig]);
    const float4 xb = *reinterpret_cast<const float4*>(&sc.Gq0[rb][4 * tig]);
    const float qa[4] = {cq0[0] + xa.x, cq1[0] + xa.y, cq0[1] + xa.z, cq1[1] + xa.w};
    const float qb[4] = {cq0[2] + xb.x, cq1[2] + xb.y, cq0[3] + xb.z, cq1[3] + xb.w};
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = ra + hr;
      const float* v = hr == 0 ? qa : qb;
      float m4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) m4[u] = (4 * tig + u <= i) ? v[u] : 0.f;
      if (kBwd && rev) {
        // row j holds column j of qscale * Aqk (the K-major B of dO^T P)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint16_t hi, lo;
          split_bf16(m4[u] * qscale, hi, lo);
          const uint32_t o = ns_off(4 * tig + u, i);
          *reinterpret_cast<uint16_t*>(sm.AQhi + o) = hi;
          *reinterpret_cast<uint16_t*>(sm.AQlo + o) = lo;
        }
      } else {
        uint32_t h0, l0, h1, l1;
        split_bf16x2(m4[0], m4[1], h0, l0);
        split_bf16x2(m4[2], m4[3], h1, l1);
        const uint32_t o = ns_off(i, 4 * tig);
        *reinterpret_cast<uint2*>(sm.AQhi + o) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(sm.AQlo + o) = make_uint2(l0, l1);
      }
    }
    // rows of the v tile past the end of the sequence: zero
    if (partial && v_used) {
      for (int idx = lane; idx < (kChunk - nv) * 16; idx += 32) {
        const int r = nv + idx / 16, c16 = idx % 16;
        *reinterpret_cast<uint4*>(st.V + (c16 >> 3) * 2048 + r * 128 + (c16 & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  pair_bar(pair);
  // ---- W = Tm (kh*2^G) for this warp's 64 channels (bf16 warp MMA, Tm split hi + lo), -W over kh*2^G
  uint32_t ahi[4], alo[4];
  {
    const int mat = lane >> 3, rr = lane & 7;
    const uint32_t moff = (uint32_t)((mat & 1) * 256 + (mat >> 1) * 128 + rr * 16);
    ldmatrix_x4(ahi, smem_u32(sm.TPhi) + moff);
    ldmatrix_x4(alo, smem_u32(sm.TPlo) + moff);
  }
#pragma unroll 2
  for (int nt = 8 * w; nt < 8 * w + 8; nt += 2) {
    uint32_t bfr[4], bfl[4];
    {
      // matrices: (tokens 0-7, tile nt), (8-15, nt), (0-7, nt+1), (8-15, nt+1)
      const int mat = lane >> 3, rr = lane & 7;
      const int row = (mat & 1) * 8 + rr;
      const int t = nt + (mat >> 1);
      ldmatrix_x4_trans(bfr, smem_u32(st.X[t >> 3]) + sw_off(row, t & 7));
      if (kPrecise) ldmatrix_x4_trans(bfl, smem_u32(wl + 2048 * (t >> 3)) + sw_off(row, t & 7));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int t = nt + u;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t bb[2] = {bfr[2 * u], bfr[2 * u + 1]};
      mma_bf16_16x8x16(d, ahi, bb);
      mma_bf16_16x8x16(d, alo, bb);
      uint8_t* xb = st.X[t >> 3];
      if (kPrecise) {   // W from kh*2^G = hi + lo, and -W written as hi (X) + lo (WL)
        const uint32_t bl[2] = {bfl[2 * u], bfl[2 * u + 1]};
        mma_bf16_16x8x16(d, ahi, bl);
        uint32_t h0, l0, h1, l1;
        split_bf16x2(-d[0], -d[1], h0, l0);
        split_bf16x2(-d[2], -d[3], h1, l1);
        uint8_t* lb = wl + 2048 * (t >> 3);
        *reinterpret_cast<uint32_t*>(xb + sw_off(gid, t & 7) + 4 * tig) = h0;
        *reinterpret_cast<uint32_t*>(xb + sw_off(gid + 8, t & 7) + 4 * tig) = h1;
        *reinterpret_cast<uint32_t*>(lb + sw_off(gid, t & 7) + 4 * tig) = l0;
        *reinterpret_cast<uint32_t*>(lb + sw_off(gid + 8, t & 7) + 4 * tig) = l1;
      } else {
        *reinterpret_cast<uint32_t*>(xb + sw_off(gid, t & 7) + 4 * tig) = pack_bf16x2(-d[0], -d[1]);
        *reinterpret_cast<uint32_t*>(xb + sw_off(gid + 8, t & 7) + 4 * tig) = pack_bf16x2(-d[2], -d[3]);
      }
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// The body of one CTA's run.  kAux: the correction and transition runs (outputs added to the
// ones already written; the run stops once its state is exactly zero); forward and reverse runs
// take the body without that code.
template <int kFlags, bool kAux>
__device__ __forceinline__ void chain_run(const ChainParams& p, const WorkItem& it) {
  // K = V = 128 is a compile-time shape; the kChainPadded variant reads K = 64 or V = 64 from p
  constexpr bool kPadded = kFlags & kChainPadded;
  constexpr bool kPrecise = kFlags & kChainPrecise;
  constexpr bool kBwd = kFlags & kChainBwd;   // the backward's storing forward runs and reverse runs
  using SmemLayout = SmemLayoutT<kPrecise>;
  using StageT = typename std::conditional<kPrecise, StagePrecise, Stage>::type;
  constexpr uint32_t kCols = kPrecise ? kTmemColsPrecise : kTmemCols;
  const int kdim = kPadded ? p.kdim : 128;    // key channels the caller's tensors hold
  const int vrows = kPadded ? p.vrows : 128;  // state rows of a chain the caller's tensors hold
  const int nchunks = (it.len + kChunk - 1) / kChunk;
  // a reverse run walks the chunks last first: iteration c handles chunk dchunk(c) of the run
  const bool rev = kBwd && (it.mode == kModeReverse || it.mode == kModeReverseCorrect);
  auto dchunk = [&](int c) { return rev ? nchunks - 1 - c : c; };
  // work items count heads x value blocks: V = 128 * vsplit columns are independent
  // chains of 128 state rows each, sharing the head's q, k, g and beta
  const int head = it.head / p.vsplit, vblk = it.head - head * p.vsplit;
  const size_t vstride = vrows == 64 ? 64 : (size_t)p.vsplit * kDimV;   // V

  extern __shared__ uint8_t smem_dyn[];
  SmemLayout& S = *reinterpret_cast<SmemLayout*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_full[kStages], bar_op_full[kStages],
      bar_d1_full[2], bar_d2_full, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ volatile int s_nz[2][4];   // per chunk parity: epilogue warp q4 saw a nonzero state

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  AbortState ab{&s_abort, p.err};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_op_full[i], 2);   // both warps of a prologue pair
    }
    mbar_init(&bar_d1_full[0], 1);
    mbar_init(&bar_d1_full[1], 1);
    mbar_init(&bar_d2_full, 1);
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp >= kWarpProlog0 && warp < kWarpEpi0) {
    const int t = threadIdx.x - kWarpProlog0 * 32;   // 0..127
    // with V = 64 the v tile's second 64 columns are never loaded: zero for the whole run
    // (128 threads x 16 bytes = the 2 KiB half-tile of each stage)
    if (vrows == 64)
      for (int s = 0; s < kStages; ++s)
        reinterpret_cast<uint4*>(S.st[s].V + 2048)[t] = make_uint4(0u, 0u, 0u, 0u);
    // with K = 64 the q, k and g tiles' channels 64-127 are never loaded: zero (the prologue
    // then writes zeros there as the gated operands of those channels)
    if (kdim == 64)
      for (int s = 0; s < kStages; ++s) {
        reinterpret_cast<uint4*>(S.st[s].X[1])[t] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(S.st[s].X[1] + 2048)[t] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(S.st[s].K + 2048)[t] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(S.st[s].G + 2048)[t] = make_uint4(0u, 0u, 0u, 0u);
      }
    // rows 16..31 of the [Tm ; 0] operands stay zero for the whole run
    if (t < 64) {
      for (int s = 0; s < kStages; ++s) {
        reinterpret_cast<uint64_t*>(S.sm[s].TPhi + 512)[t] = 0ull;
        reinterpret_cast<uint64_t*>(S.sm[s].TPlo + 512)[t] = 0ull;
      }
    }
    fence_proxy_async_smem();
  }
  if (warp == kWarpEpi0) tmem_alloc(&s_tmem, kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (nchunks > 0) {
    if (warp < kWarpEpi0) {
      // ------------------------------------------------------------ prologue
      const int pw = warp - kWarpProlog0;
      const int pair = pw >> 1, w = pw & 1;      // pair 0: even chunks, pair 1: odd chunks
      PairScratch& sc = S.ps[pair];
      const int h = head;
      const int H = p.H;
      constexpr bool gate_pre = kFlags & kGatePreactivated;   // then A_log and dt_bias may be null
      constexpr bool gate_sp = kFlags & kGateSoftplus;
      const float rate = gate_pre ? 0.f : expf(p.A_log[h]);
      // the gate's scale terms: the sigmoid gate takes -exp(A_log) log2(e) (g + dt_bias) and
      // lower_bound log2(e); the softplus gate log2(e) (g + dt_bias) and -exp(A_log)
      const float nr = gate_pre ? 0.f : (gate_sp ? kLog2e : -rate * kLog2e);
      // the head's dt_bias (K values).  With K = 64, warp 1 of a pair holds channels 64-127
      // (zero q, k and g): it reads the head's own 64 values again, and a zero output scale
      // gives those channels the decay 1 whatever they are
      const bool kpad = kdim == 64 && w == 1;
      const float* dtb = gate_pre ? nullptr : p.dt_bias + (kpad ? h * 64 - 64 : h * kdim);
      const float lbl2 = kpad ? 0.f : (gate_sp ? -rate : p.lower_bound * kLog2e);
      const int gid = lane >> 2;
      auto load_beta = [&](int c, float& b0, float& b1) {
        const int base = it.row0 + dchunk(c) * kChunk;
        const int nv = min(kChunk, it.len - dchunk(c) * kChunk);
        b0 = (c < nchunks && 2 * gid < nv) ? bf16_bits_to_f32(p.beta[(size_t)(base + 2 * gid) * H + h]) : 0.f;
        b1 = (c < nchunks && 2 * gid + 1 < nv) ? bf16_bits_to_f32(p.beta[(size_t)(base + 2 * gid + 1) * H + h])
                                               : 0.f;
      };
      float bl0, bl1;
      load_beta(pair, bl0, bl1);
      int iter = 0;
      for (int c = pair; c < nchunks; c += 2, ++iter) {
        const int s = c % kStages;
        const int nv = min(kChunk, it.len - dchunk(c) * kChunk);
        const float cb0 = bl0, cb1 = bl1;
        load_beta(c + 2, bl0, bl1);
        // both warps of the pair agree on going on (the pair shares named barriers)
        const bool okw = __all_sync(0xffffffffu, mbar_wait(&bar_full[s], (c / kStages) & 1, ab));
        if (lane == 0) sc.okf[iter & 1][w] = okw ? 1 : 0;
        pair_bar(pair);
        if (!(sc.okf[iter & 1][0] && sc.okf[iter & 1][1])) break;
        uint8_t* wl = nullptr;
        if constexpr (kPrecise) wl = &S.st[s].WL[0][0];
        prologue_pair_chunk<kFlags & kValidFlags, kPrecise, kBwd>(S.st[s], wl, S.sm[s], sc, pair, w, nv, p.err, nr,
                                                                  lbl2, dtb, cb0, cb1, lane,
                                                                  it.mode == kModeForward || rev, rev, p.scale);
        if (lane == 0) mbar_arrive(&bar_op_full[s]);
      }
    } else {
      // ------------------------------------------------------------ epilogue
      // Four warps, one TMEM lane quarter each (row v of S^T per thread).  Lane 0
      // of warp kWarpEpi0 issues every tcgen05 MMA right after a named barrier of
      // the four warps, and the TMA loads of each stage once the MMAs that read the
      // stage's previous chunk have completed; the prologue never waits on the tensor core.
      const int q4 = warp & 3;
      const int vrow = q4 * 32 + lane;
      const bool leader = (warp == kWarpEpi0) && (lane == 0);
      const uint32_t loff = static_cast<uint32_t>(q4 * 32) << 16;
      const uint32_t tS = tmem + kColState + loff;
      const uint32_t tSb = tmem + kColSbf + loff;
      const uint32_t tSlo = tmem + kColSlo + loff;   // precise runs only
      const uint32_t tD1 = tmem + kColD1 + loff;
      const int h = head;
      const size_t srow = ((size_t)it.seq * p.H + h) * vstride + (size_t)kDimV * vblk + vrow;   // state row (n, h, v)
      // the correction and transition runs take v as zero (no U); the transition writes no outputs
      const bool with_u = !kAux && it.mode == kModeForward;
      const bool with_o = !kBwd && it.mode != kModeTransition;   // the backward's runs store no outputs
      // (the backward's correction runs: kModeCorrect forward, kModeReverseCorrect reverse)
      const bool correct = kAux && (it.mode == kModeCorrect || it.mode == kModeReverseCorrect);
      // both v-free runs stop once their state is exactly zero (it then stays zero)
      constexpr bool track_zero = kAux;
      // the backward's runs store, per chunk slot, the state copy and the Vn read-out
      uint16_t* const save_state = rev ? p.save_ds1 : p.save_s0;
      float* const save_vec = rev ? p.save_dvn : p.save_vn;
      const size_t slot0 = (size_t)it.seq + (size_t)(it.row0 >> 4);   // slot of the run's chunk 0
      // instruction and shared-memory descriptors (stage s adds s * sizeof(Stage))
      const uint32_t id_u = idesc_bf16_f32(128, 32, 1, 0);
      const uint32_t id_x = idesc_bf16_f32(128, 32, 0, 0);
      const uint32_t id_s = idesc_bf16_f32(128, 128, 0, 1);   // kfac is an MN-major B
      const uint32_t id_o = idesc_bf16_f32(128, 16, 0, 0);
      const uint32_t id_w = idesc_bf16_f32(128, 16, 0, 0);   // precise: -W's remainder, Vn columns only
      // reverse runs: dO^T (MN-major A) against P^T (K-major B, N = 16); the dS^T copy against
      // K_d (K-major B, N = 16); dO^T against scale Q_p (MN-major B, N = 128)
      const uint32_t id_r1 = idesc_bf16_f32(128, 16, 1, 0);
      const uint32_t id_r2 = idesc_bf16_f32(128, 16, 0, 0);
      const uint32_t id_r3 = idesc_bf16_f32(128, 128, 1, 1);
      constexpr uint64_t kStageStep = sizeof(StageT) >> 4;
      constexpr uint64_t kSmallStep = sizeof(StageSmall) >> 4;
      const StageT& s0 = S.st[0];
      const StageSmall& m0 = S.sm[0];
      // U = V^T Tm^T of chunk c into D1[c & 1] (the leader thread only)
      auto issue_u = [&](int c) {
        const uint64_t so = (uint64_t)(c % kStages) * kStageStep;
        const uint64_t sso = (uint64_t)(c % kStages) * kSmallStep;
        const uint32_t d1 = tmem + kColD1 + 32u * (c & 1);
        const uint64_t d_v = smem_desc(smem_u32(s0.V), 2048, 1024, kSwizzle128B) + so;
        mma_ss(d1, d_v, smem_desc(smem_u32(m0.TPhi), 128, 256, kSwizzleNone) + sso, id_u, 0);
        mma_ss(d1, d_v, smem_desc(smem_u32(m0.TPlo), 128, 256, kSwizzleNone) + sso, id_u, 1);
      };
      // U, then the S-side GEMM of chunk c into D1[c & 1]
      auto issue_gemm1 = [&](int c) {
        const uint64_t so = (uint64_t)(c % kStages) * kStageStep;
        const uint32_t d1 = tmem + kColD1 + 32u * (c & 1);
        if (kBwd && rev) {
          // dVn^T = dO^T (scale P) + dS^T K_d^T into D1[c & 1] columns 0-15
          if constexpr (!kAux) {   // a correction run takes dout as zero
            const uint64_t sso = (uint64_t)(c % kStages) * kSmallStep;
            const uint64_t d_o = smem_desc(smem_u32(s0.V), 2048, 1024, kSwizzle128B) + so;
            mma_ss(d1, d_o, smem_desc(smem_u32(m0.AQhi), 128, 256, kSwizzleNone) + sso, id_r1, 0);
            mma_ss(d1, d_o, smem_desc(smem_u32(m0.AQlo), 128, 256, kSwizzleNone) + sso, id_r1, 1);
          }
          const uint64_t d_k0 = smem_desc(smem_u32(s0.K), 16, 1024, kSwizzle128B) + so;
          const uint64_t d_k1 = smem_desc(smem_u32(s0.K) + 2048, 16, 1024, kSwizzle128B) + so;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(d1, tmem + kColSbf + 8u * k, (k < 4 ? d_k0 : d_k1) + (uint64_t)((k & 3) * 2), id_r2,
                   (kAux && k == 0) ? 0u : 1u);
          tc_commit(&bar_d1_full[c & 1]);
          return;
        }
        if (with_u) issue_u(c);
        const uint64_t d_x0 = smem_desc(smem_u32(s0.X[0]), 16, 1024, kSwizzle128B) + so;
        const uint64_t d_x1 = smem_desc(smem_u32(s0.X[1]), 16, 1024, kSwizzle128B) + so;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bx = (k < 4 ? d_x0 : d_x1) + (uint64_t)((k & 3) * 2);
          mma_ts(d1, tmem + kColSbf + 8u * k, bx, id_x, (with_u || k > 0) ? 1u : 0u);
          if constexpr (kPrecise) {   // S^T = hi + lo against [-W | qh 2^G], and hi against -W's remainder
            const uint64_t bl = smem_desc(smem_u32(s0.WL[k >> 2]), 16, 1024, kSwizzle128B) + so +
                                (uint64_t)((k & 3) * 2);
            mma_ts(d1, tmem + kColSlo + 8u * k, bx, id_x, 1u);
            mma_ts(d1, tmem + kColSbf + 8u * k, bl, id_w, 1u);
          }
        }
        tc_commit(&bar_d1_full[c & 1]);
      };
      // rank-16 state update and the intra-chunk output term of chunk c
      auto issue_update = [&](int c) {
        const uint64_t so = (uint64_t)(c % kStages) * kStageStep;
        const uint64_t sso = (uint64_t)(c % kStages) * kSmallStep;
        const uint32_t d1 = tmem + kColD1 + 32u * (c & 1);
        const uint64_t a_hi = smem_desc(smem_u32(S.vn_hi), 128, 256, kSwizzleNone);
        const uint64_t a_lo = smem_desc(smem_u32(S.vn_lo), 128, 256, kSwizzleNone);
        if (kBwd && rev) {
          // dS^T += dO^T (scale Q_p) + dVn^T (-W): Q_p and -W are rows 16-31 and 0-15 of the two
          // 64-channel X tiles, 4096 bytes apart
          const uint64_t d_w = smem_desc(smem_u32(s0.X[0]), 4096, 1024, kSwizzle128B) + so;
          if constexpr (!kAux) {
            const uint64_t d_o = smem_desc(smem_u32(s0.V), 2048, 1024, kSwizzle128B) + so;
            const uint64_t d_q = smem_desc(smem_u32(s0.X[0]) + 2048, 4096, 1024, kSwizzle128B) + so;
            mma_ss(tmem + kColState, d_o, d_q, id_r3, 1);
          }
          mma_ss(tmem + kColState, a_hi, d_w, id_s, 1);
          mma_ss(tmem + kColState, a_lo, d_w, id_s, 1);
          tc_commit(&bar_d2_full);
          return;
        }
        const uint64_t kf_hi = smem_desc(smem_u32(s0.K), 2048, 1024, kSwizzle128B) + so;
        const uint64_t kf_lo = smem_desc(smem_u32(s0.G), 2048, 1024, kSwizzle128B) + so;
        mma_ss(tmem + kColState, a_hi, kf_hi, id_s, 1);
        mma_ss(tmem + kColState, a_hi, kf_lo, id_s, 1);
        mma_ss(tmem + kColState, a_lo, kf_hi, id_s, 1);
        if (with_o) {
          const uint64_t aq_hi = smem_desc(smem_u32(m0.AQhi), 128, 256, kSwizzleNone) + sso;
          const uint64_t aq_lo = smem_desc(smem_u32(m0.AQlo), 128, 256, kSwizzleNone) + sso;
          mma_ss(d1 + 16, a_hi, aq_hi, id_o, 1);
          mma_ss(d1 + 16, a_lo, aq_hi, id_o, 1);
          mma_ss(d1 + 16, a_hi, aq_lo, id_o, 1);
        }
        tc_commit(&bar_d2_full);   // every MMA of chunk c: its stage may be refilled after this
      };
      // TMA loads of chunk c into stage c % kStages (lane 0 of warp kWarpTma only)
      const bool tma_thread = (warp == kWarpTma) && (lane == 0);
      const bool load_v = with_u || (rev && !kAux);   // a reverse run loads dout where v goes
      int tma_issued = 0;
      auto issue_tma = [&](int c) {
        const int s = c % kStages;
        const int row = it.row0 + dchunk(c) * kChunk;
        Stage& st = S.st[s];
        const uint32_t qkg_bytes = kdim == 64 ? 6144u : 12288u;
        mbar_arrive_expect_tx(&bar_full[s], qkg_bytes + (load_v ? (vrows == 64 ? 2048u : 4096u) : 0u));
        // q: one 64-channel half into each S-side operand tile; k, g, v: both halves at once
        // (K = 64: one 64-channel tile of each)
        tma_load_3d(st.X[0] + 2048, &p.tm_q, &bar_full[s], 0, head, row);
        if (kdim == 64) {
          tma_load_3d(st.K, &p.tm_k, &bar_full[s], 0, head, row);
          tma_load_3d(st.G, &p.tm_g, &bar_full[s], 0, head, row);
        } else {
          tma_load_3d(st.X[1] + 2048, &p.tm_q, &bar_full[s], 64, head, row);
          tma_load_4d(st.K, &p.tm_k, &bar_full[s], 0, head, row, 0);
          tma_load_4d(st.G, &p.tm_g, &bar_full[s], 0, head, row, 0);
        }
        if (load_v) {
          if (vrows == 64) tma_load_3d(st.V, &p.tm_v, &bar_full[s], 0, head, row);   // V = 64: one tile
          else if (kBwd && rev) tma_load_4d(st.V, &p.tm_dout, &bar_full[s], 0, head, row, 0);
          else tma_load_4d(st.V, &p.tm_v, &bar_full[s], 0, head, row, 2 * vblk);
        }
        ++tma_issued;
      };
      if (tma_thread) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_g);
        tma_prefetch_desc(kBwd && rev ? &p.tm_dout : &p.tm_v);
        for (int c = 0; c < kStages && c < nchunks; ++c) issue_tma(c);
      }
      __syncwarp();
      // A correction launch may have started beside the kernel that writes its entering states
      // (and after the one that wrote the outputs it adds to).  The loads above read inputs
      // only; the epilogue warps, the only ones that read a state slot or touch the outputs,
      // wait for that kernel here (a no-op in a launch that did not overlap its predecessor).
      if constexpr (kAux) griddep_wait();
      bool issued_any = false;
      // every epilogue warp runs every named barrier below, also after an abort,
      // so that the group never waits on a warp that left early
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_op_full[0], 0, ab));
      // ---- initial state row v of S^T -> bf16 copy + decayed fp32 accumulator (a reverse run
      //      starts from dL/d final_state, fp32)
      const void* const init_ptr = rev ? static_cast<const void*>(p.dfinal) : p.init_state;
      const int init_dt = rev ? 2 : p.init_dtype;
      if (ok) {
        const StageSmall& st0 = S.sm[0];
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          float s[32];
          if (it.in_slot == kInIdentity) {
#pragma unroll
            for (int t = 0; t < 32; ++t) s[t] = (32 * j + t == vrow) ? 1.f : 0.f;
          } else if (it.in_slot >= 0) {
            const float4* src = reinterpret_cast<const float4*>(p.ws_states + (size_t)it.in_slot * 16384 +
                                                                (size_t)vrow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 x = src[t];
              s[4 * t] = x.x; s[4 * t + 1] = x.y; s[4 * t + 2] = x.z; s[4 * t + 3] = x.w;
            }
          } else if (it.in_slot == kInUser && init_ptr != nullptr && init_dt == 2 && vrow < vrows &&
                     32 * j < kdim) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(init_ptr) +
                                                                srow * kdim + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 x = src[t];
              s[4 * t] = x.x; s[4 * t + 1] = x.y; s[4 * t + 2] = x.z; s[4 * t + 3] = x.w;
            }
          } else if (it.in_slot == kInUser && init_ptr != nullptr && init_dt == 1 && vrow < vrows &&
                     32 * j < kdim) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(init_ptr) +
                                                              srow * kdim + 32 * j);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint4 x = src[t];
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                s[8 * t + 2 * u] = bf16lo_to_f32(w[u]);
                s[8 * t + 2 * u + 1] = bf16hi_to_f32(w[u]);
              }
            }
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) s[t] = 0.f;
          }
          uint32_t pk[16];
          if constexpr (kPrecise) {
            uint32_t pl[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) split_bf16x2(s[2 * t], s[2 * t + 1], pk[t], pl[t]);
            tmem_st16(tSlo + 16u * j, pl);
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(s[2 * t], s[2 * t + 1]);
          }
          tmem_st16(tSb + 16u * j, pk);
          if constexpr (kBwd) {
            uint16_t* cp = save_state + ((slot0 + dchunk(0)) * p.H + h) * 16384;
            if constexpr (kAux) add_to_copy(cp, vrow, j, s);
            else store_packed16(cp, vrow, j, pk);
          }
          uint32_t sv[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) sv[t] = __float_as_uint(s[t] * st0.gamC[32 * j + t]);
          tmem_st32(tS + 32u * j, sv);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_bar(kBarEpi, 128);
      if (leader && !s_abort) {
        tc_fence_after();
        if (mbar_wait(&bar_full[0], 0, ab)) {
          issue_gemm1(0);
          issued_any = true;
        }
      }
      __syncwarp();
      // Final state of the run's last chunk, column group j of row vrow: a workspace slot, or the
      // caller's tensor in its dtype.  A correction run adds its local final state (aux slot).
      auto write_final = [&](int j, uint32_t (&r)[32]) {
        if constexpr (kBwd) {
          // a reverse correction adds the segment's own reverse run's final dS (aux slot); a run
          // ending at a segment boundary leaves its state in a workspace slot; a reverse run that
          // reaches the sequence's start writes dL/d initial_state (fp32)
          if (correct && it.aux_slot >= 0) {
            const float4* a = reinterpret_cast<const float4*>(p.ws_states + (size_t)it.aux_slot * 16384 +
                                                              (size_t)vrow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 x = a[t];
              r[4 * t] = __float_as_uint(__uint_as_float(r[4 * t]) + x.x);
              r[4 * t + 1] = __float_as_uint(__uint_as_float(r[4 * t + 1]) + x.y);
              r[4 * t + 2] = __float_as_uint(__uint_as_float(r[4 * t + 2]) + x.z);
              r[4 * t + 3] = __float_as_uint(__uint_as_float(r[4 * t + 3]) + x.w);
            }
          }
          float4* dst = nullptr;
          if (it.out_slot >= 0)
            dst = reinterpret_cast<float4*>(p.ws_states + (size_t)it.out_slot * 16384 + (size_t)vrow * 128 + 32 * j);
          else if (rev && it.out_slot == kOutUser && p.dh0 != nullptr)
            dst = reinterpret_cast<float4*>(p.dh0 + srow * 128 + 32 * j);
          if (dst != nullptr) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[t] = make_float4(__uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                                   __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
          }
          return;
        }
        if (correct && it.aux_slot >= 0) {
          const float4* a = reinterpret_cast<const float4*>(p.ws_states + (size_t)it.aux_slot * 16384 +
                                                            (size_t)vrow * 128 + 32 * j);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 x = a[t];
            r[4 * t] = __float_as_uint(__uint_as_float(r[4 * t]) + x.x);
            r[4 * t + 1] = __float_as_uint(__uint_as_float(r[4 * t + 1]) + x.y);
            r[4 * t + 2] = __float_as_uint(__uint_as_float(r[4 * t + 2]) + x.z);
            r[4 * t + 3] = __float_as_uint(__uint_as_float(r[4 * t + 3]) + x.w);
          }
        }
        if (it.out_slot >= 0) {
          float4* dst = reinterpret_cast<float4*>(p.ws_states + (size_t)it.out_slot * 16384 +
                                                  (size_t)vrow * 128 + 32 * j);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            dst[t] = make_float4(__uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                                 __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
        } else if (it.out_slot == kOutUser && p.final_state != nullptr && p.final_dtype == 2 && vrow < vrows &&
                   32 * j < kdim) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.final_state) + srow * kdim + 32 * j);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            dst[t] = make_float4(__uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                                 __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
        } else if (it.out_slot == kOutUser && p.final_state != nullptr && p.final_dtype == 1 && vrow < vrows &&
                   32 * j < kdim) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.final_state) + srow * kdim + 32 * j);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * t]), __uint_as_float(r[8 * t + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * t + 2]), __uint_as_float(r[8 * t + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * t + 4]), __uint_as_float(r[8 * t + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * t + 6]), __uint_as_float(r[8 * t + 7])));
        }
      };
      bool stopped = false;   // a correction or transition run whose state became exactly zero
      // A backward correction run reads back, per chunk, the Vn rows and the state copy its
      // part's run stored (read-modify-writes on the chain's critical path): this thread's rows
      // of them are requested into L2 a chunk ahead (Vn of chunk c, the copy entering chunk c + 1,
      // at the top of chunk c - 1)
      auto prefetch_rows = [&](int c) {
        if constexpr (kBwd && kAux) {
          if (c < nchunks) {
            const float* vd = save_vec + ((slot0 + dchunk(c)) * p.H + h) * 2048 + vrow;
#pragma unroll
            for (int t = 0; t < 16; ++t) prefetch_l2(vd + 128 * t);
          }
          if (c + 1 < nchunks) {
            const uint16_t* cp = save_state + ((slot0 + dchunk(c + 1)) * p.H + h) * 16384;
#pragma unroll
            for (int q = 0; q < 16; ++q) prefetch_l2(cp + ((size_t)q * 128 + vrow) * 8);
          }
        }
      };
      prefetch_rows(0);
      for (int c = 0; c < nchunks; ++c) {
        const int b = c & 1;
        const int nv = min(kChunk, it.len - c * kChunk);
        const bool last = (c == nchunks - 1);
        prefetch_rows(c + 1);
        // ---- E1: Vn^T row v (16 tokens) -> split bf16 operand; then the update MMAs
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar_d1_full[b], (c >> 1) & 1, ab));
        if (ok) {
          tc_fence_after();
          uint32_t r[16];
          tmem_ld16(tD1 + 32u * b, r);
          tmem_ld_wait();
          if constexpr (kBwd) {   // Vn (dVn) of this chunk, [16 tokens][128 v]; a correction adds its part
            float* vd = save_vec + ((slot0 + dchunk(c)) * p.H + h) * 2048 + vrow;
            if constexpr (kAux) {
              float old[16];
#pragma unroll
              for (int t = 0; t < 16; ++t) old[t] = vd[128 * t];
#pragma unroll
              for (int t = 0; t < 16; ++t) vd[128 * t] = old[t] + __uint_as_float(r[t]);
            } else {
#pragma unroll
              for (int t = 0; t < 16; ++t) vd[128 * t] = __uint_as_float(r[t]);
            }
          }
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int t = 0; t < 8; ++t)
            split_bf16x2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1]), hw[t], lw[t]);
          *reinterpret_cast<uint4*>(S.vn_hi + ns_off(vrow, 0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(S.vn_hi + ns_off(vrow, 8)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          *reinterpret_cast<uint4*>(S.vn_lo + ns_off(vrow, 0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          *reinterpret_cast<uint4*>(S.vn_lo + ns_off(vrow, 8)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar(kBarEpi, 128);
        if (leader && !s_abort) {
          tc_fence_after();
          issue_update(c);
        }
        __syncwarp();
        // ---- E2: the new state S' -> bf16 copy (A operand of the next S-side GEMM) and,
        //      in the same pass, the fp32 accumulator decayed by the next chunk's 2^G_C
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar_d2_full, c & 1, ab));
        if (!last)
          ok = ok && __all_sync(0xffffffffu,
                                mbar_wait(&bar_op_full[(c + 1) % kStages], ((c + 1) / kStages) & 1, ab));
        uint32_t nz = 0u;   // any nonzero bit of S' in this thread's row
        if (ok) {
          tc_fence_after();
          const StageSmall& stn = S.sm[(c + 1) % kStages];
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld32(tS + 32u * j, r);
            tmem_ld_wait();
            if (!last) {
              if (track_zero) {
#pragma unroll
                for (int t = 0; t < 32; ++t) nz |= r[t] & 0x7fffffffu;
              }
              uint32_t pk[16];
              if constexpr (kPrecise) {
                uint32_t pl[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                  split_bf16x2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1]), pk[t], pl[t]);
                tmem_st16(tSlo + 16u * j, pl);
              } else {
#pragma unroll
                for (int t = 0; t < 16; ++t)
                  pk[t] = pack_bf16x2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1]));
              }
              tmem_st16(tSb + 16u * j, pk);
              if constexpr (kBwd) {   // the state entering the next chunk handled (S_0, or dS_1 in reverse)
                uint16_t* cp = save_state + ((slot0 + dchunk(c + 1)) * p.H + h) * 16384;
                if constexpr (kAux) {
                  float sv[32];
#pragma unroll
                  for (int t = 0; t < 32; ++t) sv[t] = __uint_as_float(r[t]);
                  add_to_copy(cp, vrow, j, sv);
                } else {
                  store_packed16(cp, vrow, j, pk);
                }
              }
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const float4 gm = *reinterpret_cast<const float4*>(&stn.gamC[32 * j + 4 * t]);
                float a0 = __uint_as_float(r[4 * t]), a1 = __uint_as_float(r[4 * t + 1]);
                float a2 = __uint_as_float(r[4 * t + 2]), a3 = __uint_as_float(r[4 * t + 3]);
                fmul2(a0, a1, gm.x, gm.y);
                fmul2(a2, a3, gm.z, gm.w);
                r[4 * t] = __float_as_uint(a0);
                r[4 * t + 1] = __float_as_uint(a1);
                r[4 * t + 2] = __float_as_uint(a2);
                r[4 * t + 3] = __float_as_uint(a3);
              }
              tmem_st32(tS + 32u * j, r);
            } else {
              write_final(j, r);
            }
          }
          if (!last) tmem_st_wait();
        }
        // Zero vote of the four epilogue warps.  Every warp writes its entry (a warp that has
        // given up votes nonzero), so all four take the same decision after the barrier below.
        if (track_zero && !last) {
          const int any_nz = __any_sync(0xffffffffu, nz != 0u) ? 1 : 0;
          if (lane == 0) s_nz[b][q4] = ok ? any_nz : 1;
        }
        tc_fence_before();
        named_bar(kBarEpi, 128);
        const bool stop_now =
            track_zero && !last && (s_nz[b][0] | s_nz[b][1] | s_nz[b][2] | s_nz[b][3]) == 0;
        if (stop_now && leader) s_abort = 1;   // no error: it tells the other roles to unwind
        if (!last && !stop_now && leader && !s_abort) {
          tc_fence_after();
          const int c1 = c + 1;
          if (mbar_wait(&bar_full[c1 % kStages], (c1 / kStages) & 1, ab)) issue_gemm1(c1);
        }
        // stage c % kStages is free: this warp saw every MMA of chunk c complete (bar_d2_full)
        if (tma_thread && ok && !stop_now && !s_abort && c + kStages < nchunks) issue_tma(c + kStages);
        __syncwarp();
        // ---- outputs of this chunk (overlaps the next S-side GEMM): each warp stages its
        //      32 output columns of the 16 token rows in shared memory, then writes them as
        //      16-byte pieces, four per row (64 contiguous bytes).  A correction run adds its
        //      term to the outputs its segment's forward run wrote.
        if (with_o && ok) {
          uint32_t r[16];
          tmem_ld16(tD1 + 32u * b + 16u, r);
          tmem_ld_wait();
          const size_t row_elems = (size_t)p.H * vstride;
          uint16_t* obase = p.out + ((size_t)(it.row0 + c * kChunk) * p.H + h) * vstride + (size_t)kDimV * vblk;
          if (correct) {
            // (unrolled with a guard: a loop bound of nv would index r at run time and put it
            // in local memory for every mode).  Every output is read before any is written:
            // the compiler cannot tell that the stores do not alias the later loads, and would
            // otherwise wait for each load in turn.
            if (vrow < vrows) {
              uint16_t old[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) old[i] = i < nv ? obase[(size_t)i * row_elems + vrow] : (uint16_t)0;
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (i < nv)
                  obase[(size_t)i * row_elems + vrow] = __bfloat16_as_ushort(
                      __float2bfloat16_rn(bf16_bits_to_f32(old[i]) + p.scale * __uint_as_float(r[i])));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              *reinterpret_cast<uint16_t*>(&S.ostage[i][2 * vrow]) =
                  __bfloat16_as_ushort(__float2bfloat16_rn(p.scale * __uint_as_float(r[i])));
            __syncwarp();
            if ((reinterpret_cast<uintptr_t>(p.out) & 15u) == 0) {
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const int q = lane + 32 * rr, i = q >> 2, seg = q & 3;
                if (i < nv && 32 * q4 < vrows)
                  *reinterpret_cast<uint4*>(obase + (size_t)i * row_elems + 32 * q4 + 8 * seg) =
                      *reinterpret_cast<const uint4*>(&S.ostage[i][64 * q4 + 16 * seg]);
              }
            } else {
              for (int i = 0; i < nv && vrow < vrows; ++i)
                obase[(size_t)i * row_elems + vrow] = *reinterpret_cast<const uint16_t*>(&S.ostage[i][2 * vrow]);
            }
            __syncwarp();   // the staging rows are rewritten by the next chunk
          }
        }
        if (stop_now) {   // uniform across the four warps
          stopped = true;
          break;
        }
      }
      // a correction run that stopped early ends with a zero difference: its final state is
      // the local one from its aux slot
      if (stopped && correct && it.out_slot != kOutNone) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = 0u;
          write_final(j, r);
        }
      }
      // a transition run records whether it ended exactly zero (then its slot is not written)
      if (it.mode == kModeTransition && leader && it.out_slot >= 0)
        p.zero_flags[it.out_slot] = stopped ? 1 : 0;
      const bool unwind = s_abort || stopped;
      if (leader && unwind && issued_any) {  // wait for MMAs in flight before TMEM is released
        tc_commit(&bar_drain);
        mbar_wait_drain(&bar_drain, 0);
      }
      if (tma_thread && unwind) {  // let loads in flight land before the CTA exits
        for (int c = (tma_issued > kStages ? tma_issued - kStages : 0); c < tma_issued; ++c)
          mbar_wait_drain(&bar_full[c % kStages], (c / kStages) & 1);
      }
      __syncwarp();
    }
  } else if (warp >= kWarpEpi0) {
    // zero-length run: the final state equals the initial state
    if constexpr (kAux) griddep_wait();
    const int q4 = warp & 3;
    const int vrow = q4 * 32 + lane;
    if constexpr (kBwd) {   // a reverse run: dL/d initial_state = dL/d final_state
      if (rev && it.out_slot == kOutUser && p.dh0 != nullptr) {
        const size_t srow = ((size_t)it.seq * p.H + head) * 128 + vrow;
        for (int t = 0; t < 128; ++t)
          p.dh0[srow * 128 + t] = (it.in_slot == kInUser && p.dfinal != nullptr) ? p.dfinal[srow * 128 + t] : 0.f;
      }
    } else {
      if (it.mode == kModeTransition && threadIdx.x == kWarpEpi0 * 32 && it.out_slot >= 0)
        p.zero_flags[it.out_slot] = 0;   // the identity
      const size_t srow = ((size_t)it.seq * p.H + head) * vstride + (size_t)kDimV * vblk + vrow;
      for (int t = 0; t < 128; ++t) {
        float x = 0.f;
        if (it.in_slot == kInIdentity) x = (t == vrow) ? 1.f : 0.f;
        else if (it.in_slot >= 0) x = p.ws_states[(size_t)it.in_slot * 16384 + (size_t)vrow * 128 + t];
        else if (it.in_slot == kInUser && p.init_state && p.init_dtype == 2 && vrow < vrows && t < kdim)
          x = static_cast<const float*>(p.init_state)[srow * kdim + t];
        else if (it.in_slot == kInUser && p.init_state && p.init_dtype == 1 && vrow < vrows && t < kdim)
          x = bf16_bits_to_f32(static_cast<const uint16_t*>(p.init_state)[srow * kdim + t]);
        if (it.mode == kModeCorrect && it.aux_slot >= 0) x += p.ws_states[(size_t)it.aux_slot * 16384 + (size_t)vrow * 128 + t];
        if (it.out_slot >= 0) p.ws_states[(size_t)it.out_slot * 16384 + (size_t)vrow * 128 + t] = x;
        else if (it.out_slot == kOutUser && p.final_state && p.final_dtype == 2 && vrow < vrows && t < kdim)
          static_cast<float*>(p.final_state)[srow * kdim + t] = x;
        else if (it.out_slot == kOutUser && p.final_state && p.final_dtype == 1 && vrow < vrows && t < kdim)
          static_cast<uint16_t*>(p.final_state)[srow * kdim + t] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpEpi0) tmem_dealloc(tmem, kCols);
}

// kFlags (steps the caller already did) is a template parameter: the prologue's inner
// loops then carry no per-element tests of it
// Two CTAs per SM (128 registers a thread); the precise-state kernels run one per SM.
template <int kFlags>
__global__ void __launch_bounds__(kThreads, (kFlags & kChainPrecise) ? 1 : 2)
    kda_chain_kernel(const __grid_constant__ ChainParams p) {
  // Item of this CTA.  The forward launch pairs runs by SM: the list is longest first, the
  // first CTA to start on an SM takes the longest run left and the second the shortest, so
  // a long chain shares its SM with a short one and then runs alone.
  // the segment scan's transition runs let the forward runs' launch start beside them
  // and the backward's runs let its correction launch start beside them
  if constexpr ((kFlags & (kChainAux | kChainBwd)) != 0) griddep_launch_dependents();
  int item = blockIdx.x;
  if (p.take != nullptr) {
    __shared__ int s_item;
    if (threadIdx.x == 0) {
      const int n_items = *p.item_count;
      int pick = -1;
      if (atomicAdd(&p.take[0], 1) < n_items) {   // at most n_items picks: head and tail never meet
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        const int arrival = atomicAdd(&p.sm_arrivals[smid % kMaxSmIds], 1);
        pick = (arrival & 1) == 0 ? atomicAdd(&p.take[1], 1) : n_items - 1 - atomicAdd(&p.take[2], 1);
      }
      s_item = pick;
    }
    __syncthreads();
    item = s_item;
  } else if (item >= *p.item_count) {
    item = -1;
  }
  // a launch that overlapped the transition runs completes only after them: every CTA waits
  // for the previous kernel before it exits (the composition after this launch reads both)
  if (item >= 0) {
    const WorkItem it = p.items[item];
    if (it.len >= 0) chain_run<kFlags, (kFlags & kChainAux) != 0>(p, it);   // len < 0: a placeholder
  }
  griddep_wait();
}

// Launch of one family of kernel variants: kBase is 0 (the usual kernels) or kChainPrecise, each
// with or without kChainAux (the correction and transition runs' kernels).
// Entries: the caller-side flags (the preactivated and softplus gates exclude each other: no
// kernel for both), then the same for K = 64 or V = 64 (kChainPadded).
template <int kBase>
cudaError_t launch_chain_table(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev = false) {
  using Kernel = void (*)(ChainParams);
  static constexpr Kernel kernels[32] = {
      kda_chain_kernel<kBase + 0>, kda_chain_kernel<kBase + 1>, kda_chain_kernel<kBase + 2>,
      kda_chain_kernel<kBase + 3>, kda_chain_kernel<kBase + 4>, kda_chain_kernel<kBase + 5>,
      kda_chain_kernel<kBase + 6>, kda_chain_kernel<kBase + 7>, kda_chain_kernel<kBase + 8>, nullptr,
      kda_chain_kernel<kBase + 10>, nullptr, kda_chain_kernel<kBase + 12>, nullptr,
      kda_chain_kernel<kBase + 14>, nullptr,
      kda_chain_kernel<kBase + 16>, kda_chain_kernel<kBase + 17>, kda_chain_kernel<kBase + 18>,
      kda_chain_kernel<kBase + 19>, kda_chain_kernel<kBase + 20>, kda_chain_kernel<kBase + 21>,
      kda_chain_kernel<kBase + 22>, kda_chain_kernel<kBase + 23>, kda_chain_kernel<kBase + 24>, nullptr,
      kda_chain_kernel<kBase + 26>, nullptr, kda_chain_kernel<kBase + 28>, nullptr,
      kda_chain_kernel<kBase + 30>, nullptr};
  constexpr size_t smem = chain_smem_bytes_t<(kBase & kChainPrecise) != 0>();
  // the shared-memory opt-in is a per-device setting: made once per device
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    for (Kernel k : kernels) {
      if (k == nullptr) continue;
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  if (grid <= 0) return cudaSuccess;
  const bool padded = p.kdim != 128 || p.vrows != 128;
  const Kernel k = kernels[(p.flags & kValidFlags) | (padded ? kChainPadded : 0)];
  if (k == nullptr) return cudaErrorInvalidValue;
  if (!overlap_prev) {
    k<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace kda
