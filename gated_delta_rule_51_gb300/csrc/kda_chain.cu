// kda_chain.cu -- the fused chunked KDA forward kernel for sm_103a.
//
// One CTA walks one run of 16-token chunks of one (sequence, head) -- a whole
// sequence, or one segment of a long one -- and keeps the 128 x 128 fp32 state
// on chip for the whole run (FlashKDA: "processes 16-token chunks", "FP32 FMA
// instructions for state updates").  Per chunk, with S the state on entry:
//
//   G    = within-chunk inclusive cumsum of the base-2 log-decay (per channel)
//   Akk  = tril(beta_i * (kh*2^G)(kh*2^-G)^T, -1)   Aqk = tril((qh*2^G)(kh*2^-G)^T, 0)
//   Tm   = (I + Akk)^-1 Diag(beta)          (forward substitution, fp32)
//   W    = Tm (kh*2^G),  U = Tm v,  Vn = U - W S
//   O    = scale * ((qh*2^G) S + Aqk Vn)
//   S'   = Diag(2^G_C) S + (kh*2^(G_C-G))^T Vn
//
// Warp roles (320 threads):
//   warp 0      TMA producer: q, k, g tiles into a ring, v tile into the
//               operand stage (v is the A operand of U^T = V^T Tm^T as is).
//   warp 1      tcgen05 issuer (one thread).  State GEMMs in the M = V = 128
//               orientation:  D1 = V^T Tm^T + S^T [-W^T | (qh 2^G)^T]   (N = 32)
//                             D2 += Vn^T kfac ;  D1[:,16:] += Vn^T Aqk^T
//   warps 2-5   prologue: gate, cumsum, L2 norms, Gram matrices (warp MMA,
//               tf32), inverse, W (warp MMA, split bf16), operand tiles.
//   warps 6-9   epilogue: Vn read-out (split into bf16 hi + lo), outputs,
//               state decay + bf16 copy of S^T for the next chunk's A operand.
// TMEM (256 columns): [0,128) S^T fp32 accumulator, [128,192) S^T as packed
// bf16 (A operand read straight from TMEM), [192,256) two 32-column D1 tiles.
//
// Precision: the S-side GEMM runs on bf16 copies of S^T, W and qh*2^G; the
// rank-16 state update, U and Aqk*Vn use a split-bf16 (hi + lo) scheme, and
// the Grams use tf32, which keeps the fp32 state within ~1e-6 of exact.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kThreads = 320;
constexpr int kNRaw = 2;
constexpr int kNOp = 2;
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpProlog0 = 2;
constexpr int kWarpEpi0 = 6;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColState = 0;
constexpr uint32_t kColSbf = 128;
constexpr uint32_t kColD1 = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kBarProlog = 1;   // named barrier id of the prologue warps

struct RawStage {         // q, k, g tiles, each 2 boxes [16 rows x 64 ch] bf16 SW128
  uint8_t q[4096];
  uint8_t k[4096];
  uint8_t g[4096];
};
struct OpStage {
  uint8_t X[8192];        // B of the S-GEMM: rows 0-15 = -W, rows 16-31 = qh*2^G; K-major SW128
  uint8_t v[4096];        // v tile from TMA (MN-major SW128 A operand)
  uint8_t KFhi[4096];     // kfac^T [128 ch][16 tok] K-major, no swizzle (hi part)
  uint8_t KFlo[4096];
  uint8_t TPhi[1024];     // [Tm ; 0] [32 rows][16] K-major, no swizzle
  uint8_t TPlo[1024];
  uint8_t AQhi[512];      // Aqk [16][16] K-major, no swizzle
  uint8_t AQlo[512];
  float gamC[128];        // 2^G_C per channel
  uint8_t pad[24576 - 8192 - 4096 - 8192 - 2048 - 1024 - 512];
};
static_assert(sizeof(OpStage) == 24576, "op stage size");
struct PrologScratch {
  uint16_t kg[16][136];        // bf16 kh*2^G, row stride 272 B (ldmatrix friendly)
  float gram[4][2][16][16];    // per-warp partial Grams (kk, qk)
  float normp[4][16][2];       // per-warp partial |q|^2, |k|^2
  float beta[16];
  float pad[12];
};
struct SmemLayout {
  RawStage raw[kNRaw];
  OpStage op[kNOp];
  uint8_t vn_hi[4096];         // Vn^T [128 v][16 tok] K-major, no swizzle
  uint8_t vn_lo[4096];
  PrologScratch ps;
};

size_t chain_smem_bytes() { return sizeof(SmemLayout) + 1024; }

// byte offset of element (row r, channel c) in a [16 x 128] bf16 tile stored as
// two TMA boxes of [16 x 64] with the 128-byte swizzle
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 6) * 2048 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}
// byte offset of (row n, k) in a K-major SW128 [32 x 128] bf16 operand (two 4 KB k-blocks)
__device__ __forceinline__ uint32_t xop_off(int n, int c) {
  return (uint32_t)((c >> 6) * 4096 + (n >> 3) * 1024 + (n & 7) * 128 + ((((c & 63) >> 3) ^ (n & 7)) << 4) +
                    (c & 7) * 2);
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

__global__ void __launch_bounds__(kThreads, 2) kda_chain_kernel(const __grid_constant__ ChainParams p) {
  if ((int)blockIdx.x >= *p.item_count) return;
  const WorkItem it = p.items[blockIdx.x];
  if (it.len < 0) return;   // placeholder entry of a work list
  const int nchunks = (it.len + kChunk - 1) / kChunk;

  extern __shared__ uint8_t smem_dyn[];
  SmemLayout& S = *reinterpret_cast<SmemLayout*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bar_full[kNRaw], bar_raw_empty[kNRaw], bar_op_full[kNOp],
      bar_op_empty[kNOp], bar_d1_full[2], bar_vn_ready, bar_d2_full, bar_s_ready, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  AbortState ab{&s_abort, p.err};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNRaw; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_raw_empty[i], 1);
    }
    for (int i = 0; i < kNOp; ++i) {
      mbar_init(&bar_op_full[i], 1);
      mbar_init(&bar_op_empty[i], 1);
    }
    mbar_init(&bar_d1_full[0], 1);
    mbar_init(&bar_d1_full[1], 1);
    mbar_init(&bar_vn_ready, 4);
    mbar_init(&bar_d2_full, 1);
    mbar_init(&bar_s_ready, 4);
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp >= kWarpProlog0 && warp < kWarpEpi0) {
    // rows 16..31 of the [Tm ; 0] operands stay zero for the whole run
    const int t = threadIdx.x - kWarpProlog0 * 32;
    for (int s = 0; s < kNOp; ++s) {
      reinterpret_cast<uint32_t*>(S.op[s].TPhi + 512)[t] = 0u;
      reinterpret_cast<uint32_t*>(S.op[s].TPlo + 512)[t] = 0u;
    }
    fence_proxy_async_smem();
  }
  if (warp == kWarpProducer) tmem_alloc(&s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (nchunks > 0) {
    if (warp == kWarpProducer) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_g);
        tma_prefetch_desc(&p.tm_v);
        const bool load_v = it.mode != kModeTransition;
        int issued = 0;
        for (int c = 0; c < nchunks; ++c) {
          const int rs = c % kNRaw, os = c % kNOp;
          if (c >= kNRaw && !mbar_wait(&bar_raw_empty[rs], ((c / kNRaw) - 1) & 1, ab)) break;
          if (c >= kNOp && !mbar_wait(&bar_op_empty[os], ((c / kNOp) - 1) & 1, ab)) break;
          const int row = it.row0 + c * kChunk;
          mbar_arrive_expect_tx(&bar_full[rs], load_v ? 16384u : 12288u);
          for (int b = 0; b < 2; ++b) {
            tma_load_3d(S.raw[rs].q + b * 2048, &p.tm_q, &bar_full[rs], b * 64, it.head, row);
            tma_load_3d(S.raw[rs].k + b * 2048, &p.tm_k, &bar_full[rs], b * 64, it.head, row);
            tma_load_3d(S.raw[rs].g + b * 2048, &p.tm_g, &bar_full[rs], b * 64, it.head, row);
            if (load_v) tma_load_3d(S.op[os].v + b * 2048, &p.tm_v, &bar_full[rs], b * 64, it.head, row);
          }
          ++issued;
        }
        if (s_abort) {  // let loads in flight land before the CTA exits
          for (int c = (issued > kNRaw ? issued - kNRaw : 0); c < issued; ++c)
            mbar_wait_drain(&bar_full[c % kNRaw], (c / kNRaw) & 1);
        }
      }
      __syncwarp();
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t id_u = idesc_bf16_f32(128, 32, 1, 0);
        const uint32_t id_x = idesc_bf16_f32(128, 32, 0, 0);
        const uint32_t id_s = idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t id_o = idesc_bf16_f32(128, 16, 0, 0);
        const uint32_t vnh = smem_u32(S.vn_hi), vnl = smem_u32(S.vn_lo);
        const bool with_u = it.mode != kModeTransition;
        const bool with_o = it.mode == kModeForward;
        bool issued_any = false;
        for (int c = 0; c < nchunks; ++c) {
          const int rs = c % kNRaw, os = c % kNOp, b = c & 1;
          const uint32_t d1 = tmem + kColD1 + 32u * b;
          OpStage& op = S.op[os];
          if (!mbar_wait(&bar_op_full[os], (c / kNOp) & 1, ab)) break;
          if (!mbar_wait(&bar_full[rs], (c / kNRaw) & 1, ab)) break;
          tc_fence_after();
          if (with_u) {
            const uint64_t a_v = smem_desc(smem_u32(op.v), 2048, 1024, kSwizzle128B);
            mma_ss(d1, a_v, smem_desc(smem_u32(op.TPhi), 128, 256, kSwizzleNone), id_u, 0);
            mma_ss(d1, a_v, smem_desc(smem_u32(op.TPlo), 128, 256, kSwizzleNone), id_u, 1);
          }
          issued_any = true;
          if (!mbar_wait(&bar_s_ready, c & 1, ab)) break;
          tc_fence_after();
          const uint32_t xb = smem_u32(op.X);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint64_t bd = smem_desc(xb + (s >> 2) * 4096 + (s & 3) * 32, 16, 1024, kSwizzle128B);
            mma_ts(d1, tmem + kColSbf + 8u * s, bd, id_x, (with_u || s > 0) ? 1u : 0u);
          }
          tc_commit(&bar_d1_full[b]);
          if (!mbar_wait(&bar_vn_ready, c & 1, ab)) break;
          tc_fence_after();
          const uint64_t a_hi = smem_desc(vnh, 128, 256, kSwizzleNone);
          const uint64_t a_lo = smem_desc(vnl, 128, 256, kSwizzleNone);
          const uint64_t kf_hi = smem_desc(smem_u32(op.KFhi), 128, 256, kSwizzleNone);
          const uint64_t kf_lo = smem_desc(smem_u32(op.KFlo), 128, 256, kSwizzleNone);
          mma_ss(tmem + kColState, a_hi, kf_hi, id_s, 1);
          mma_ss(tmem + kColState, a_hi, kf_lo, id_s, 1);
          mma_ss(tmem + kColState, a_lo, kf_hi, id_s, 1);
          if (with_o) {
            const uint64_t aq_hi = smem_desc(smem_u32(op.AQhi), 128, 256, kSwizzleNone);
            const uint64_t aq_lo = smem_desc(smem_u32(op.AQlo), 128, 256, kSwizzleNone);
            mma_ss(d1 + 16, a_hi, aq_hi, id_o, 1);
            mma_ss(d1 + 16, a_lo, aq_hi, id_o, 1);
            mma_ss(d1 + 16, a_hi, aq_lo, id_o, 1);
          }
          tc_commit(&bar_d2_full);
          tc_commit(&bar_op_empty[os]);
        }
        if (s_abort && issued_any) {  // wait for MMAs in flight before TMEM is released
          tc_commit(&bar_drain);
          mbar_wait_drain(&bar_drain, 0);
        }
      }
      __syncwarp();
    } else if (warp < kWarpEpi0) {
      // ------------------------------------------------------------ prologue
      const int pw = warp - kWarpProlog0;        // channels [32 pw, 32 pw + 32)
      const int ptid = threadIdx.x - kWarpProlog0 * 32;
      const int gid = lane >> 2, tig = lane & 3;
      PrologScratch& ps = S.ps;
      const int h = it.head;
      const int H = p.H;
      // per-thread channel constants: ch(pp, e) = 32 pw + 8 pp + 2 tig + e
      const float rate = expf(p.A_log[h]);
      const float nr = -rate * kLog2e;
      float nrdb[4][2];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
#pragma unroll
        for (int e = 0; e < 2; ++e) nrdb[pp][e] = nr * p.dt_bias[h * kDimK + 32 * pw + 8 * pp + 2 * tig + e];
      const float lbl2 = p.lower_bound * kLog2e;
      // beta logits for rows gid, gid + 8 of the current chunk (prefetched one chunk ahead)
      auto load_beta = [&](int c, float& b0, float& b1) {
        const int base = it.row0 + c * kChunk;
        const int nv = min(kChunk, it.len - c * kChunk);
        b0 = (c < nchunks && gid < nv) ? bf16_bits_to_f32(p.beta[(size_t)(base + gid) * H + h]) : 0.f;
        b1 = (c < nchunks && gid + 8 < nv) ? bf16_bits_to_f32(p.beta[(size_t)(base + gid + 8) * H + h]) : 0.f;
      };
      float bl0, bl1;
      load_beta(0, bl0, bl1);
      for (int c = 0; c < nchunks; ++c) {
        const int rs = c % kNRaw, os = c % kNOp;
        const int nv = min(kChunk, it.len - c * kChunk);
        OpStage& op = S.op[os];
        const float cur_b0 = bl0, cur_b1 = bl1;
        load_beta(c + 1, bl0, bl1);
        bool ok = mbar_wait(&bar_full[rs], (c / kNRaw) & 1, ab);
        if (c >= kNOp) ok = mbar_wait(&bar_op_empty[os], ((c / kNOp) - 1) & 1, ab) && ok;
        ok = __all_sync(0xffffffffu, ok);
        // ---- load q, k, g for rows gid and gid + 8 (pairs of channels)
        float q[2][4][2], k[2][4][2], g[2][4][2];
        if (ok) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = gid + 8 * hr;
            const bool valid = r < nv;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
              const uint32_t off = tile_off(r, 32 * pw + 8 * pp + 2 * tig);
              const uint32_t wq = *reinterpret_cast<const uint32_t*>(S.raw[rs].q + off);
              const uint32_t wk = *reinterpret_cast<const uint32_t*>(S.raw[rs].k + off);
              const uint32_t wg = *reinterpret_cast<const uint32_t*>(S.raw[rs].g + off);
              q[hr][pp][0] = valid ? bf16lo_to_f32(wq) : 0.f;
              q[hr][pp][1] = valid ? bf16hi_to_f32(wq) : 0.f;
              k[hr][pp][0] = valid ? bf16lo_to_f32(wk) : 0.f;
              k[hr][pp][1] = valid ? bf16hi_to_f32(wk) : 0.f;
              g[hr][pp][0] = bf16lo_to_f32(wg);
              g[hr][pp][1] = bf16hi_to_f32(wg);
            }
          }
          // partial squared norms over this thread's 8 channels, then over tig
          float sq[2], sk[2];
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            sq[hr] = 0.f;
            sk[hr] = 0.f;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                sq[hr] = fmaf(q[hr][pp][e], q[hr][pp][e], sq[hr]);
                sk[hr] = fmaf(k[hr][pp][e], k[hr][pp][e], sk[hr]);
              }
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {
              sq[hr] += __shfl_xor_sync(0xffffffffu, sq[hr], m);
              sk[hr] += __shfl_xor_sync(0xffffffffu, sk[hr], m);
            }
          }
          if (tig == 0) {
            ps.normp[pw][gid][0] = sq[0];
            ps.normp[pw][gid][1] = sk[0];
            ps.normp[pw][gid + 8][0] = sq[1];
            ps.normp[pw][gid + 8][1] = sk[1];
          }
        }
        named_bar(kBarProlog, 128);
        if (ptid == 0 && ok) mbar_arrive(&bar_raw_empty[rs]);   // q, k, g are in registers now
        float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
        float gc_l2[4][2];
        if (ok) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = gid + 8 * hr;
            float tq = 0.f, tk = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              tq += ps.normp[w][r][0];
              tk += ps.normp[w][r][1];
            }
            rq[hr] = rsqrt_approx(tq + 1e-6f);
            rk[hr] = rsqrt_approx(tk + 1e-6f);
          }
          // ---- gate: base-2 log-decay per element, then the within-chunk cumsum over rows
#pragma unroll
          for (int pp = 0; pp < 4; ++pp)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float a = 0.f, bq = 0.f;
              {
                const float t0 = ex2_approx(fmaf(nr, g[0][pp][e], nrdb[pp][e]));
                const float t1 = ex2_approx(fmaf(nr, g[1][pp][e], nrdb[pp][e]));
                a = (gid < nv) ? lbl2 * rcp_approx(1.f + t0) : 0.f;
                bq = (gid + 8 < nv) ? lbl2 * rcp_approx(1.f + t1) : 0.f;
              }
#pragma unroll
              for (int d = 1; d <= 4; d <<= 1) {
                const float ya = __shfl_up_sync(0xffffffffu, a, 4 * d);
                const float yb = __shfl_up_sync(0xffffffffu, bq, 4 * d);
                if (gid >= d) {
                  a += ya;
                  bq += yb;
                }
              }
              bq += __shfl_sync(0xffffffffu, a, 28 + tig);
              gc_l2[pp][e] = __shfl_sync(0xffffffffu, bq, 28 + tig);
              g[0][pp][e] = a;    // g now holds G (base 2) for rows gid, gid + 8
              g[1][pp][e] = bq;
            }
        }
        // ---- decay-scaled operands, Gram partials (tf32 warp MMA), operand tiles
        float kgv[2][4][2], kiv[2][4][2];
        if (ok) {
          float ck0[4] = {0, 0, 0, 0}, ck1[4] = {0, 0, 0, 0}, cq0[4] = {0, 0, 0, 0}, cq1[4] = {0, 0, 0, 0};
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            float qg[2][2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float G = g[hr][pp][e];
                const float gam = ex2_approx(G);
                const float ginv = ex2_approx(-G);
                const float kh = k[hr][pp][e] * rk[hr];
                kgv[hr][pp][e] = kh * gam;
                kiv[hr][pp][e] = kh * ginv;
                qg[hr][e] = q[hr][pp][e] * rq[hr] * gam;
              }
            const uint32_t ak[4] = {f32_to_tf32(kgv[0][pp][0]), f32_to_tf32(kgv[1][pp][0]),
                                    f32_to_tf32(kgv[0][pp][1]), f32_to_tf32(kgv[1][pp][1])};
            const uint32_t aq[4] = {f32_to_tf32(qg[0][0]), f32_to_tf32(qg[1][0]), f32_to_tf32(qg[0][1]),
                                    f32_to_tf32(qg[1][1])};
            const uint32_t b0[2] = {f32_to_tf32(kiv[0][pp][0]), f32_to_tf32(kiv[0][pp][1])};
            const uint32_t b1[2] = {f32_to_tf32(kiv[1][pp][0]), f32_to_tf32(kiv[1][pp][1])};
            mma_tf32_16x8x8(ck0, ak, b0);
            mma_tf32_16x8x8(ck1, ak, b1);
            mma_tf32_16x8x8(cq0, aq, b0);
            mma_tf32_16x8x8(cq1, aq, b1);
            // qh*2^G -> rows 16..31 of X; kh*2^G (bf16) -> scratch for W
            const int ch = 32 * pw + 8 * pp + 2 * tig;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int r = gid + 8 * hr;
              *reinterpret_cast<uint32_t*>(op.X + xop_off(16 + r, ch)) = pack_bf16x2(qg[hr][0], qg[hr][1]);
              *reinterpret_cast<uint32_t*>(&ps.kg[r][ch]) = pack_bf16x2(kgv[hr][pp][0], kgv[hr][pp][1]);
            }
            // kfac = kh * 2^(G_C - G) as split bf16, transposed K-major [ch][tok]
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float gcl = ex2_approx(gc_l2[pp][e]);
              if (gid == 0) op.gamC[ch + e] = gcl;
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                uint16_t hi, lo;
                split_bf16(kiv[hr][pp][e] * gcl, hi, lo);
                const uint32_t o = ns_off(ch + e, gid + 8 * hr);
                *reinterpret_cast<uint16_t*>(op.KFhi + o) = hi;
                *reinterpret_cast<uint16_t*>(op.KFlo + o) = lo;
              }
            }
          }
          // partial Grams -> scratch
          {
            float* gk = &ps.gram[pw][0][0][0];
            float* gq = &ps.gram[pw][1][0][0];
            const int c0 = 2 * tig;
            *reinterpret_cast<float2*>(gk + gid * 16 + c0) = make_float2(ck0[0], ck0[1]);
            *reinterpret_cast<float2*>(gk + (gid + 8) * 16 + c0) = make_float2(ck0[2], ck0[3]);
            *reinterpret_cast<float2*>(gk + gid * 16 + 8 + c0) = make_float2(ck1[0], ck1[1]);
            *reinterpret_cast<float2*>(gk + (gid + 8) * 16 + 8 + c0) = make_float2(ck1[2], ck1[3]);
            *reinterpret_cast<float2*>(gq + gid * 16 + c0) = make_float2(cq0[0], cq0[1]);
            *reinterpret_cast<float2*>(gq + (gid + 8) * 16 + c0) = make_float2(cq0[2], cq0[3]);
            *reinterpret_cast<float2*>(gq + gid * 16 + 8 + c0) = make_float2(cq1[0], cq1[1]);
            *reinterpret_cast<float2*>(gq + (gid + 8) * 16 + 8 + c0) = make_float2(cq1[2], cq1[3]);
          }
          if (pw == 0 && tig == 0) {
            ps.beta[gid] = (gid < nv) ? rcp_approx(1.f + ex2_approx(-cur_b0 * kLog2e)) : 0.f;
            ps.beta[gid + 8] = (gid + 8 < nv) ? rcp_approx(1.f + ex2_approx(-cur_b1 * kLog2e)) : 0.f;
          }
        }
        named_bar(kBarProlog, 128);
        // ---- warp 0 of the prologue: reduce Grams, invert, write Tm and Aqk
        if (ok && pw == 0) {
          // reduce the four partials in place into gram[0]
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int e = lane + 32 * i;   // 0..511 over [2][16][16]
            float* base = &ps.gram[0][0][0][0];
            const float s = base[e] + base[512 + e] + base[1024 + e] + base[1536 + e];
            base[e] = s;
          }
          __syncwarp();
          const float* Gk = &ps.gram[0][0][0][0];
          const float* Gq = &ps.gram[0][1][0][0];
          if (lane < 16) {
            // column j = lane of X = (I + Akk)^-1, Akk[i][m] = beta_i Gk[i][m] (m < i)
            const int j = lane;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m) {
#pragma unroll
              for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-ps.beta[i] * Gk[i * 16 + m], x[m], x[i]);
            }
            const float bj = ps.beta[j];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint16_t hi, lo;
              split_bf16(x[i] * bj, hi, lo);
              const uint32_t o = ns_off(i, j);
              *reinterpret_cast<uint16_t*>(op.TPhi + o) = hi;
              *reinterpret_cast<uint16_t*>(op.TPlo + o) = lo;
            }
          } else {
            // Aqk row i = lane - 16, inclusive lower triangle
            const int i = lane - 16;
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int jj = 0; jj < 16; jj += 2) {
              uint16_t h0, l0, h1, l1;
              split_bf16(jj <= i ? Gq[i * 16 + jj] : 0.f, h0, l0);
              split_bf16(jj + 1 <= i ? Gq[i * 16 + jj + 1] : 0.f, h1, l1);
              hw[jj / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
              lw[jj / 2] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
            *reinterpret_cast<uint4*>(op.AQhi + ns_off(i, 0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(op.AQhi + ns_off(i, 8)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            *reinterpret_cast<uint4*>(op.AQlo + ns_off(i, 0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            *reinterpret_cast<uint4*>(op.AQlo + ns_off(i, 8)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
          }
        }
        named_bar(kBarProlog, 128);
        // ---- W = Tm (kh*2^G) for this warp's 32 channels (bf16 warp MMA, Tm split hi + lo)
        if (ok) {
          uint32_t ahi[4], alo[4];
          {
            const int mat = lane >> 3, rr = lane & 7;
            const uint32_t moff = (uint32_t)((mat & 1) * 256 + (mat >> 1) * 128 + rr * 16);
            ldmatrix_x4(ahi, smem_u32(op.TPhi) + moff);
            ldmatrix_x4(alo, smem_u32(op.TPlo) + moff);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t bfr[4];
            {
              const int mat = lane >> 3, rr = lane & 7;
              const int krow = (mat & 1) * 8 + rr;
              const int ncol = 32 * pw + 16 * half + 8 * (mat >> 1);
              ldmatrix_x4_trans(bfr, smem_u32(&ps.kg[krow][ncol]));
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              float d[4] = {0.f, 0.f, 0.f, 0.f};
              const uint32_t bb[2] = {bfr[2 * nt], bfr[2 * nt + 1]};
              mma_bf16_16x8x16(d, ahi, bb);
              mma_bf16_16x8x16(d, alo, bb);
              const int ch = 32 * pw + 16 * half + 8 * nt + 2 * tig;
              *reinterpret_cast<uint32_t*>(op.X + xop_off(gid, ch)) = pack_bf16x2(-d[0], -d[1]);
              *reinterpret_cast<uint32_t*>(op.X + xop_off(gid + 8, ch)) = pack_bf16x2(-d[2], -d[3]);
            }
          }
          // zero the rows of the v tile that lie past the end of the sequence
          if (nv < kChunk && it.mode != kModeTransition) {
            for (int idx = ptid; idx < (kChunk - nv) * 16; idx += 128) {
              const int r = nv + idx / 16, cchunk = idx % 16;
              *reinterpret_cast<uint4*>(op.v + (cchunk >> 3) * 2048 + r * 128 + (cchunk & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
        named_bar(kBarProlog, 128);
        if (ptid == 0 && ok) mbar_arrive(&bar_op_full[os]);
      }
    } else {
      // ------------------------------------------------------------ epilogue
      const int q4 = warp & 3;
      const int vrow = q4 * 32 + lane;
      const uint32_t loff = static_cast<uint32_t>(q4 * 32) << 16;
      const uint32_t tS = tmem + kColState + loff;
      const uint32_t tSb = tmem + kColSbf + loff;
      const uint32_t tD1 = tmem + kColD1 + loff;
      const int h = it.head;
      const size_t srow = ((size_t)it.seq * p.H + h) * kDimV + vrow;   // user state row (n, h, v)
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_op_full[0], 0, ab));
      // ---- initial state row v of S^T -> bf16 copy + decayed fp32 accumulator
      if (ok) {
        const OpStage& op0 = S.op[0];
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
          } else if (it.in_slot == kInUser && p.init_state != nullptr && p.init_dtype == 2) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.init_state) +
                                                                srow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 x = src[t];
              s[4 * t] = x.x; s[4 * t + 1] = x.y; s[4 * t + 2] = x.z; s[4 * t + 3] = x.w;
            }
          } else if (it.in_slot == kInUser && p.init_state != nullptr && p.init_dtype == 1) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.init_state) +
                                                              srow * 128 + 32 * j);
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
          if (it.aux_slot >= 0) {
            float4* dst = reinterpret_cast<float4*>(p.ws_states + (size_t)it.aux_slot * 16384 +
                                                    (size_t)vrow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t) dst[t] = make_float4(s[4 * t], s[4 * t + 1], s[4 * t + 2], s[4 * t + 3]);
          }
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(s[2 * t], s[2 * t + 1]);
          tmem_st16(tSb + 16u * j, pk);
          uint32_t sv[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) sv[t] = __float_as_uint(s[t] * op0.gamC[32 * j + t]);
          tmem_st32(tS + 32u * j, sv);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&bar_s_ready);
      for (int c = 0; c < nchunks && ok; ++c) {
        const int b = c & 1;
        const int nv = min(kChunk, it.len - c * kChunk);
        // ---- E1: Vn^T row v (16 tokens) -> split bf16 operand
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_d1_full[b], (c >> 1) & 1, ab));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t r[16];
          tmem_ld16(tD1 + 32u * b, r);
          tmem_ld_wait();
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            uint16_t h0, l0, h1, l1;
            split_bf16(__uint_as_float(r[2 * t]), h0, l0);
            split_bf16(__uint_as_float(r[2 * t + 1]), h1, l1);
            hw[t] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            lw[t] = (uint32_t)l0 | ((uint32_t)l1 << 16);
          }
          *reinterpret_cast<uint4*>(S.vn_hi + ns_off(vrow, 0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(S.vn_hi + ns_off(vrow, 8)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          *reinterpret_cast<uint4*>(S.vn_lo + ns_off(vrow, 0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          *reinterpret_cast<uint4*>(S.vn_lo + ns_off(vrow, 8)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_vn_ready);
        // ---- E2: outputs and the state for the next chunk
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_d2_full, c & 1, ab));
        if (!ok) break;
        tc_fence_after();
        if (it.mode == kModeForward) {
          uint32_t r[16];
          tmem_ld16(tD1 + 32u * b + 16u, r);
          tmem_ld_wait();
          const size_t base = ((size_t)(it.row0 + c * kChunk) * p.H + h) * kDimV + vrow;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < nv) {
              const __nv_bfloat16 o = __float2bfloat16_rn(p.scale * __uint_as_float(r[i]));
              p.out[base + (size_t)i * p.H * kDimV] = __bfloat16_as_ushort(o);
            }
          }
        }
        const bool last = (c == nchunks - 1);
        if (!last) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_op_full[(c + 1) % kNOp], ((c + 1) / kNOp) & 1, ab));
          if (!ok) break;
        }
        const OpStage& opn = S.op[(c + 1) % kNOp];
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld32(tS + 32u * j, r);
          tmem_ld_wait();
          if (!last) {
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1]));
            tmem_st16(tSb + 16u * j, pk);
#pragma unroll
            for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * opn.gamC[32 * j + t]);
            tmem_st32(tS + 32u * j, r);
          } else if (it.out_slot >= 0) {
            float4* dst = reinterpret_cast<float4*>(p.ws_states + (size_t)it.out_slot * 16384 +
                                                    (size_t)vrow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[t] = make_float4(__uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                                   __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
          } else if (it.out_slot == kOutUser && p.final_state != nullptr && p.final_dtype == 2) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.final_state) + srow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[t] = make_float4(__uint_as_float(r[4 * t]), __uint_as_float(r[4 * t + 1]),
                                   __uint_as_float(r[4 * t + 2]), __uint_as_float(r[4 * t + 3]));
          } else if (it.out_slot == kOutUser && p.final_state != nullptr && p.final_dtype == 1) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.final_state) + srow * 128 + 32 * j);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * t]), __uint_as_float(r[8 * t + 1])),
                                  pack_bf16x2(__uint_as_float(r[8 * t + 2]), __uint_as_float(r[8 * t + 3])),
                                  pack_bf16x2(__uint_as_float(r[8 * t + 4]), __uint_as_float(r[8 * t + 5])),
                                  pack_bf16x2(__uint_as_float(r[8 * t + 6]), __uint_as_float(r[8 * t + 7])));
          }
        }
        if (!last) {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_s_ready);
        }
      }
    }
  } else if (warp >= kWarpEpi0) {
    // zero-length run: the final state equals the initial state
    const int q4 = warp & 3;
    const int vrow = q4 * 32 + lane;
    const size_t srow = ((size_t)it.seq * p.H + it.head) * kDimV + vrow;
    for (int t = 0; t < 128; ++t) {
      float x = 0.f;
      if (it.in_slot == kInIdentity) x = (t == vrow) ? 1.f : 0.f;
      else if (it.in_slot >= 0) x = p.ws_states[(size_t)it.in_slot * 16384 + (size_t)vrow * 128 + t];
      else if (it.in_slot == kInUser && p.init_state && p.init_dtype == 2)
        x = static_cast<const float*>(p.init_state)[srow * 128 + t];
      else if (it.in_slot == kInUser && p.init_state && p.init_dtype == 1)
        x = bf16_bits_to_f32(static_cast<const uint16_t*>(p.init_state)[srow * 128 + t]);
      if (it.out_slot >= 0) p.ws_states[(size_t)it.out_slot * 16384 + (size_t)vrow * 128 + t] = x;
      else if (it.out_slot == kOutUser && p.final_state && p.final_dtype == 2)
        static_cast<float*>(p.final_state)[srow * 128 + t] = x;
      else if (it.out_slot == kOutUser && p.final_state && p.final_dtype == 1)
        static_cast<uint16_t*>(p.final_state)[srow * 128 + t] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpProducer) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t s) {
  const size_t smem = chain_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kda_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  kda_chain_kernel<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
