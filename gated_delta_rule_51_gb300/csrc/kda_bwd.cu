// kda_bwd.cu -- the backward pass of the KDA forward (K = V = 128): the gradients of
// L = sum(dout * out) + sum(dfinal * final_state) with respect to q, k, v, g, the beta
// logits, the initial state, A_log and dt_bias.
//
// FlashKDA's README defines the forward only ("Kernel API"); the gradient follows from
// that definition.  Per (sequence, head) the forward is the token recurrence
//     P_t = Diag(alpha_t) S_{t-1},  u_t = v_t - P_t^T kh_t,  S_t = P_t + beta_t kh_t u_t^T,
//     o_t = scale S_t^T qh_t,
// and its reverse step, for a state gradient dS (dL/dS_t), is
//     dS += scale qh dO^T;  dqh = scale S_t dO;  w = dS^T kh;  du = beta w;  dv = du;
//     dbeta = u . w;  dkh = beta dS u - P du;  dP = dS - kh du^T;
//     dalpha[c] = sum_j dP[c][j] S_{t-1}[c][j];  dS_{t-1} = Diag(alpha) dP,
// followed by the chain rule through the L2 norms, the beta sigmoid and the gate.
//
// Every value column j of S (a row of the [V, K] state layout) evolves independently given
// the per-token vectors alpha, kh, qh, beta; only dqh, dkh, dalpha and dbeta sum over
// columns.  So the recurrences split the 128 state rows of a head over four CTAs of eight
// warps, four rows a warp, each lane holding four key channels of each of its rows in
// registers (the decode step's layout), and sum the column partials in a fixed order.
// Each chunk's per-token vectors, v and dout are staged in shared memory once, so the
// per-token steps read no global memory.
//
// Two forms.  The chunked one (the default for the gate with a lower bound; "chunked path"
// below) runs the chunk recurrence on tensor cores in the chain kernels and every chunk's
// gradients in parallel:
//   items    the chains' runs (a forward and a reverse run per part of each (sequence, head));
//   (chains: kda_chain_kernel, kChainBwd, launched from kda_api.cu)
//   xprod    per chunk: dO S0^T, Vn dS1^T, dVn S0^T on bf16 warp MMA, sum_v dS1 S0;
//   chunk    per chunk: the 16 x 16 and 16 x 128 products on tf32 warp MMA (fp32-accurate
//            split), then every token's gradients and the dA_log terms;
//   param    dA_log and dt_bias summed over tokens, as below.
// The recurrent one (the other gates, or KDA_BWD_RECURRENT), in launch order:
//   prep     per token-head: alpha = exp(ghat), beta, qh, kh and the norms' scales;
//   ckpt     the forward recurrence, storing the state at every kBwdChunk-th token;
//   reverse  per chunk, last first: for each token (last first) the state before it is
//            recomputed from the chunk's stored state (or from the state before the
//            chunk's middle token, kept once per chunk), then the reverse step runs; the
//            per-token column partials of dqh, dkh, dalpha, dbeta go to the workspace;
//   finish   per token-head: the partials summed, then the norms, the sigmoid and the gate;
//   param    dA_log and dt_bias summed over tokens in blocks, then over blocks.
// Memory: the stored states take (B T / kBwdChunk + N + 1) x H x 64 KiB.  No kernel of either
// form waits on another CTA; the only barriers are __syncthreads.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = kRowsPerWarp * kWarps;   // state rows per CTA
static_assert(kRows * kBwdSlices == 128, "four CTAs cover the 128 state rows of a head");
static_assert(kThreads >= 128, "one thread per key channel in the column sums");
static_assert(kBwdRowStride % 4 == 0, "prep rows are copied as float4");

// A chunk's per-token vectors (alpha, kh, qh, beta, rq, rk) and the CTA's rows of v and
// scale * dout, staged in shared memory once per chunk by the whole CTA.
struct ChunkStage {
  float prep[kBwdChunk][kBwdRowStride];
  float v[kBwdChunk][kRows];
  float dout[kBwdChunk][kRows];
};

__device__ __forceinline__ float bfv(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float softp(float x) { return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x)); }
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 bf4(const uint16_t* p) {   // four bf16 values, 8-byte aligned
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(bfv(w.x & 0xffffu), bfv(w.x >> 16), bfv(w.y & 0xffffu), bfv(w.y >> 16));
}

// The token range of sequence n, clamped to [0, BT); a malformed cu_seqlens is flagged
// (by the caller's designated thread) and can then only give wrong values, never an
// access outside the buffers.
struct SeqRange {
  int64_t t0, len;
};
__device__ __forceinline__ SeqRange seq_range(const BwdParams& p, int n, bool flag) {
  if (p.cu == nullptr) return {(int64_t)n * p.T, p.T};
  const int64_t s = p.cu[n], e = p.cu[n + 1];
  const int64_t sc = min(max(s, (int64_t)0), p.BT), ec = min(max(e, sc), p.BT);
  if (flag && (s != sc || e != ec || (n == 0 && s != 0) || (n == p.N - 1 && e != p.BT)))
    atomicOr(p.err, kErrBadSeqlens);
  return {sc, ec - sc};
}

// ---------------------------------------------------------------------------- prep
// One warp per token-head, four channels a lane.
__global__ void __launch_bounds__(128) kda_bwd_prep_kernel(const BwdParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t TH = p.BT * p.H;
  const int64_t wstride = (int64_t)gridDim.x * 4;
  const bool gate_pre = p.flags & kGatePreactivated, gate_sp = p.flags & kGateSoftplus;
  const bool norm = !(p.flags & kNoQkL2Norm), beta_pre = p.flags & kBetaPreactivated;
  const int c0 = 4 * lane;
  for (int64_t th = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); th < TH; th += wstride) {
    const int h = (int)(th % p.H);
    const float4 q = bf4(p.q + th * 128 + c0), k = bf4(p.k + th * 128 + c0), g = bf4(p.g + th * 128 + c0);
    const float qq = warp_sum(dot4(q, q)), kk = warp_sum(dot4(k, k));
    const float rq = norm ? 1.f / sqrtf(qq + 1e-6f) : 1.f, rk = norm ? 1.f / sqrtf(kk + 1e-6f) : 1.f;
    float gv[4] = {g.x, g.y, g.z, g.w}, al[4];
    if (gate_pre) {
#pragma unroll
      for (int i = 0; i < 4; ++i) al[i] = expf(gv[i]);
    } else {
      const float rate = expf(p.A_log[h]);
      const float4 db = ld4(p.dt_bias + (size_t)h * 128 + c0);
      const float dv[4] = {db.x, db.y, db.z, db.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = gv[i] + dv[i];
        al[i] = expf(gate_sp ? -rate * softp(x) : p.lower_bound * sigm(rate * x));
      }
    }
    float* pr = p.prep + th * kBwdRowStride;
    st4(pr + c0, make_float4(al[0], al[1], al[2], al[3]));
    st4(pr + 128 + c0, make_float4(k.x * rk, k.y * rk, k.z * rk, k.w * rk));
    st4(pr + 256 + c0, make_float4(q.x * rq, q.y * rq, q.z * rq, q.w * rq));
    if (lane == 0) {
      const float braw = bfv(p.beta[th]);
      st4(pr + 384, make_float4(beta_pre ? braw : sigm(braw), rq, rk, 0.f));
    }
  }
}

// One forward step of a warp's rows for a staged token: P = alpha S; u = v - P^T kh;
// S = P + beta kh u.  pr: the token's prep row; vr: its v values of this warp's rows.
__device__ __forceinline__ void fwd_step(float4 (&S)[kRowsPerWarp], const float* pr, const float* vr, int lane) {
  const float4 al = ld4(pr + 4 * lane), kh = ld4(pr + 128 + 4 * lane);
  const float b = pr[384];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const float4 sp = make_float4(al.x * S[i].x, al.y * S[i].y, al.z * S[i].z, al.w * S[i].w);
    const float u = vr[i] - warp_sum(dot4(sp, kh));
    const float bu = b * u;
    S[i] = make_float4(sp.x + bu * kh.x, sp.y + bu * kh.y, sp.z + bu * kh.z, sp.w + bu * kh.w);
  }
}

// Staging of tokens tc .. tc + nv - 1 of head h (rows r0 .. r0 + kRows - 1 of v and dout)
// in two halves: stage_load reads a chunk into registers (issued a chunk ahead, so the
// loads are in flight while the current chunk computes), stage_store writes them to
// shared memory between two barriers.
constexpr int kPrepF4 = kBwdRowStride / 4;                                  // float4 per prep row
constexpr int kStagePasses = (kBwdChunk * kPrepF4 + kThreads - 1) / kThreads;
static_assert(kBwdChunk * kRows <= kThreads, "one v (and dout) value per thread");
struct StageRegs {
  float4 pr[kStagePasses];
  float v, d;
};

__device__ __forceinline__ void stage_load(StageRegs& R, const BwdParams& p, int64_t tc, int nv, int h, int r0,
                                           bool with_dout) {
#pragma unroll
  for (int k = 0; k < kStagePasses; ++k) {
    const int idx = threadIdx.x + k * kThreads;
    if (idx < nv * kPrepF4) {
      const int i = idx / kPrepF4, f = idx % kPrepF4;
      R.pr[k] = ld4(p.prep + ((tc + i) * p.H + h) * kBwdRowStride + 4 * f);
    }
  }
  if ((int)threadIdx.x < nv * kRows) {
    const int i = threadIdx.x / kRows, r = threadIdx.x % kRows;
    const size_t e = ((size_t)(tc + i) * p.H + h) * 128 + r0 + r;
    R.v = bfv(p.v[e]);
    R.d = with_dout ? bfv(p.dout[e]) * p.scale : 0.f;
  }
}

__device__ __forceinline__ void stage_store(ChunkStage& cs, const StageRegs& R, int nv) {
#pragma unroll
  for (int k = 0; k < kStagePasses; ++k) {
    const int idx = threadIdx.x + k * kThreads;
    if (idx < nv * kPrepF4) st4(&cs.prep[idx / kPrepF4][4 * (idx % kPrepF4)], R.pr[k]);
  }
  if ((int)threadIdx.x < nv * kRows) {
    cs.v[threadIdx.x / kRows][threadIdx.x % kRows] = R.v;
    cs.dout[threadIdx.x / kRows][threadIdx.x % kRows] = R.d;
  }
}

__device__ __forceinline__ void load_rows(float4 (&S)[kRowsPerWarp], const float* base, int lane) {
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) S[i] = ld4(base + i * 128 + 4 * lane);
}

// ---------------------------------------------------------------------------- ckpt
// Grid: N x H x kBwdSlices CTAs; warp w of slice s owns state rows 32 s + 4 w .. + 3.
__global__ void __launch_bounds__(kThreads) kda_bwd_ckpt_kernel(const BwdParams p) {
  __shared__ __align__(16) ChunkStage cs;
  const int slice = blockIdx.x % kBwdSlices, nh = blockIdx.x / kBwdSlices;
  const int n = nh / p.H, h = nh % p.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = slice * kRows, row0 = r0 + warp * kRowsPerWarp;
  const SeqRange r = seq_range(p, n, slice == 0 && threadIdx.x == 0);
  float4 S[kRowsPerWarp];
  const size_t srow = ((size_t)nh * 128 + row0) * 128;   // element offset of this warp's first row
  if (p.init_dtype == 2) {
    load_rows(S, static_cast<const float*>(p.init_state) + srow, lane);
  } else if (p.init_dtype == 1) {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) S[i] = bf4(static_cast<const uint16_t*>(p.init_state) + srow + i * 128 + 4 * lane);
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t base = r.t0 / kBwdChunk + n;   // this sequence's first stored-state slot
  const int64_t nch = (r.len + kBwdChunk - 1) / kBwdChunk;
  auto chunk_len = [&](int64_t j) { return (int)min((int64_t)kBwdChunk, r.len - j * kBwdChunk); };
  StageRegs R;
  if (nch > 0) stage_load(R, p, r.t0, chunk_len(0), h, r0, false);
  for (int64_t j = 0; j < nch; ++j) {
    const int nv = chunk_len(j);
    float* dst = p.ckpt + (((size_t)(base + j) * p.H + h) * 128 + row0) * 128;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) st4(dst + i * 128 + 4 * lane, S[i]);
    __syncthreads();   // the previous chunk's staged values are read
    stage_store(cs, R, nv);
    __syncthreads();
    if (j + 1 < nch) stage_load(R, p, r.t0 + (j + 1) * kBwdChunk, chunk_len(j + 1), h, r0, false);
    for (int i = 0; i < nv; ++i) fwd_step(S, cs.prep[i], &cs.v[i][warp * kRowsPerWarp], lane);
  }
}

// ---------------------------------------------------------------------------- reverse
__global__ void __launch_bounds__(kThreads) kda_bwd_reverse_kernel(const BwdParams p) {
  __shared__ __align__(16) float red[2][kWarps][kBwdRowStride];
  __shared__ __align__(16) ChunkStage cs;
  const int slice = blockIdx.x % kBwdSlices, nh = blockIdx.x / kBwdSlices;
  const int n = nh / p.H, h = nh % p.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = slice * kRows, row0 = r0 + warp * kRowsPerWarp;
  const SeqRange r = seq_range(p, n, false);
  const int64_t TH = p.BT * p.H;
  const size_t srow = ((size_t)nh * 128 + row0) * 128;
  float4 dS[kRowsPerWarp];
  if (p.dfinal != nullptr) {
    load_rows(dS, p.dfinal + srow, lane);
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) dS[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t base = r.t0 / kBwdChunk + n;
  const int64_t nch = (r.len + kBwdChunk - 1) / kBwdChunk;
  int par = 0;
  auto chunk_len = [&](int64_t j) { return (int)min((int64_t)kBwdChunk, r.len - j * kBwdChunk); };
  constexpr int kMid = kBwdChunk / 2;
  StageRegs R;
  if (nch > 0) stage_load(R, p, r.t0 + (nch - 1) * kBwdChunk, chunk_len(nch - 1), h, r0, true);
  for (int64_t j = nch - 1; j >= 0; --j) {
    const float* ck = p.ckpt + (((size_t)(base + j) * p.H + h) * 128 + row0) * 128;
    const int64_t tc = r.t0 + j * kBwdChunk;
    const int nv = chunk_len(j);
    __syncthreads();   // the previous chunk's staged values are read
    stage_store(cs, R, nv);
    __syncthreads();
    if (j > 0) stage_load(R, p, tc - kBwdChunk, chunk_len(j - 1), h, r0, true);
    const int wr = warp * kRowsPerWarp;   // this warp's rows within the staged ones
    // the state before the chunk's middle token, for the second half's recomputations
    float4 Sm[kRowsPerWarp];
    if (nv > kMid) {
      load_rows(Sm, ck, lane);
      for (int jj = 0; jj < kMid; ++jj) fwd_step(Sm, cs.prep[jj], &cs.v[jj][wr], lane);
    }
    for (int i = nv - 1; i >= 0; --i) {
      // the state before token tc + i, recomputed from the chunk's stored state or its middle
      float4 S[kRowsPerWarp];
      int from = 0;
      if (i >= kMid) {
#pragma unroll
        for (int ii = 0; ii < kRowsPerWarp; ++ii) S[ii] = Sm[ii];
        from = kMid;
      } else {
        load_rows(S, ck, lane);
      }
      for (int jj = from; jj < i; ++jj) fwd_step(S, cs.prep[jj], &cs.v[jj][wr], lane);
      const int64_t th = (tc + i) * p.H + h;
      const float* pr = cs.prep[i];
      const float4 al = ld4(pr + 4 * lane), kh = ld4(pr + 128 + 4 * lane), qh = ld4(pr + 256 + 4 * lane);
      const float b = pr[384];
      float4 aq = make_float4(0.f, 0.f, 0.f, 0.f), ak = aq, aa = aq;
      float dbeta = 0.f, dv_mine = 0.f;
#pragma unroll
      for (int ii = 0; ii < kRowsPerWarp; ++ii) {
        const float4 s0 = S[ii];
        const float4 sp = make_float4(al.x * s0.x, al.y * s0.y, al.z * s0.z, al.w * s0.w);
        const float u = cs.v[i][wr + ii] - warp_sum(dot4(sp, kh));
        const float bu = b * u;
        const float4 st = make_float4(sp.x + bu * kh.x, sp.y + bu * kh.y, sp.z + bu * kh.z, sp.w + bu * kh.w);
        const float d = cs.dout[i][wr + ii];   // scale * dO for this row
        aq.x += d * st.x; aq.y += d * st.y; aq.z += d * st.z; aq.w += d * st.w;
        float4 ds = dS[ii];
        ds.x += d * qh.x; ds.y += d * qh.y; ds.z += d * qh.z; ds.w += d * qh.w;
        const float w = warp_sum(dot4(ds, kh));
        const float du = b * w;
        dbeta += u * w;
        ak.x += bu * ds.x - du * sp.x; ak.y += bu * ds.y - du * sp.y;
        ak.z += bu * ds.z - du * sp.z; ak.w += bu * ds.w - du * sp.w;
        const float4 dp = make_float4(ds.x - du * kh.x, ds.y - du * kh.y, ds.z - du * kh.z, ds.w - du * kh.w);
        aa.x += dp.x * s0.x; aa.y += dp.y * s0.y; aa.z += dp.z * s0.z; aa.w += dp.w * s0.w;
        dS[ii] = make_float4(al.x * dp.x, al.y * dp.y, al.z * dp.z, al.w * dp.w);
        if (lane == ii) dv_mine = du;
      }
      if (lane < kRowsPerWarp) p.dv[th * 128 + row0 + lane] = dv_mine;
      float* rw = red[par][warp];
      st4(rw + 4 * lane, aq);
      st4(rw + 128 + 4 * lane, ak);
      st4(rw + 256 + 4 * lane, aa);
      if (lane == 0) rw[384] = dbeta;
      __syncthreads();
      if (threadIdx.x < 128) {
        // column sums over the CTA's warps, in a fixed order; one thread per channel
        const int c = threadIdx.x;
        float sq = 0.f, sk = 0.f, sa = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          sq += red[par][w][c];
          sk += red[par][w][128 + c];
          sa += red[par][w][256 + c];
        }
        float* pp = p.part + ((size_t)slice * TH + th) * kBwdRowStride;
        pp[c] = sq;
        pp[128 + c] = sk;
        pp[256 + c] = sa;
        if (c == 0) {
          float sb = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) sb += red[par][w][384];
          pp[384] = sb;
        }
      }
      par ^= 1;   // the next token writes the other buffer: one barrier per token suffices
    }
  }
  if (p.dh0 != nullptr) {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) st4(p.dh0 + srow + i * 128 + 4 * lane, dS[i]);
  }
}

// ---------------------------------------------------------------------------- finish
// One warp per token-head: the slices' partials summed in order, then the chain rule
// through the norms (dx = r (dxh - xh (xh . dxh))), the beta sigmoid and the gate.
__global__ void __launch_bounds__(128) kda_bwd_finish_kernel(const BwdParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t TH = p.BT * p.H;
  const int64_t wstride = (int64_t)gridDim.x * 4;
  const bool gate_pre = p.flags & kGatePreactivated, gate_sp = p.flags & kGateSoftplus;
  const bool norm = !(p.flags & kNoQkL2Norm), beta_pre = p.flags & kBetaPreactivated;
  const int c0 = 4 * lane;
  for (int64_t th = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); th < TH; th += wstride) {
    const int h = (int)(th % p.H);
    float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq, sa = sq;
    float sb = 0.f;
#pragma unroll
    for (int s = 0; s < kBwdSlices; ++s) {
      const float* pp = p.part + ((size_t)s * TH + th) * kBwdRowStride;
      const float4 a = ld4(pp + c0), b = ld4(pp + 128 + c0), c = ld4(pp + 256 + c0);
      sq.x += a.x; sq.y += a.y; sq.z += a.z; sq.w += a.w;
      sk.x += b.x; sk.y += b.y; sk.z += b.z; sk.w += b.w;
      sa.x += c.x; sa.y += c.y; sa.z += c.z; sa.w += c.w;
      sb += pp[384];
    }
    const float* pr = p.prep + th * kBwdRowStride;
    const float4 al = ld4(pr + c0), kh = ld4(pr + 128 + c0), qh = ld4(pr + 256 + c0);
    const float4 tail = ld4(pr + 384);   // beta, rq, rk
    float4 dq = sq, dk = sk;
    if (norm) {
      const float qd = warp_sum(dot4(qh, sq)), kd = warp_sum(dot4(kh, sk));
      dq = make_float4(tail.y * (sq.x - qd * qh.x), tail.y * (sq.y - qd * qh.y), tail.y * (sq.z - qd * qh.z),
                       tail.y * (sq.w - qd * qh.w));
      dk = make_float4(tail.z * (sk.x - kd * kh.x), tail.z * (sk.y - kd * kh.y), tail.z * (sk.z - kd * kh.z),
                       tail.z * (sk.w - kd * kh.w));
    }
    st4(p.dq + th * 128 + c0, dq);
    st4(p.dk + th * 128 + c0, dk);
    // gate: dghat = dalpha alpha
    const float dgh[4] = {sa.x * al.x, sa.y * al.y, sa.z * al.z, sa.w * al.w};
    float dg[4], wa = 0.f;
    if (gate_pre) {
#pragma unroll
      for (int i = 0; i < 4; ++i) dg[i] = dgh[i];
    } else {
      const float rate = expf(p.A_log[h]);
      const float4 g = bf4(p.g + th * 128 + c0);
      const float4 db = ld4(p.dt_bias + (size_t)h * 128 + c0);
      const float x[4] = {g.x + db.x, g.y + db.y, g.z + db.z, g.w + db.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (gate_sp) {
          // ghat = -rate softplus(x): d/dx = -rate sigmoid(x); d/dA_log = ghat
          dg[i] = dgh[i] * (-rate * sigm(x[i]));
          wa += dgh[i] * (-rate * softp(x[i]));
        } else {
          // ghat = lb sigmoid(z), z = rate x: d/dz = lb s (1 - s); d/dx = rate d/dz; d/dA_log = z d/dz
          const float z = rate * x[i], s = sigm(z);
          const float dz = dgh[i] * p.lower_bound * s * (1.f - s);
          dg[i] = dz * rate;
          wa += dz * z;
        }
      }
      wa = warp_sum(wa);
    }
    st4(p.dg + th * 128 + c0, make_float4(dg[0], dg[1], dg[2], dg[3]));
    if (lane == 0) {
      p.dbeta[th] = beta_pre ? sb : sb * tail.x * (1.f - tail.x);
      p.dA_tok[th] = wa;
    }
  }
}

// ---------------------------------------------------------------------------- params
// Grid (nblk, H): block b sums dg (= d dt_bias per token) and the dA_log terms of tokens
// [256 b, 256 b + 256) of head h; then one CTA per head sums the blocks in order.
__global__ void __launch_bounds__(128) kda_bwd_param_kernel(const BwdParams p) {
  const int blk = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int64_t t0 = (int64_t)blk * kBwdParamTokens, t1 = min(p.BT, t0 + kBwdParamTokens);
  // sixteen partial sums (token t into sum t mod 16) so that sixteen loads are in flight at once;
  // they are combined in a fixed order, so the result is the same on every run
  float a16[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) a16[u] = 0.f;
  int64_t t = t0;
  for (; t + 16 <= t1; t += 16) {
    float x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = p.dg[((t + u) * p.H + h) * 128 + c];
#pragma unroll
    for (int u = 0; u < 16; ++u) a16[u] += x[u];
  }
  for (; t < t1; ++t) a16[0] += p.dg[(t * p.H + h) * 128 + c];   // the tail, in order
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int u = 0; u < w; ++u) a16[u] += a16[u + w];
  const float acc = a16[0];
  float accA = 0.f;
  for (int64_t ta = t0 + c; ta < t1; ta += 128) accA += p.dA_tok[ta * p.H + h];
  __shared__ float sA[128];
  sA[c] = accA;
  __syncthreads();
  float* dst = p.ppart + ((size_t)blk * p.H + h) * kBwdParamStride;
  dst[c] = acc;
  if (c == 0) {
    float s = 0.f;
    for (int i = 0; i < 128; ++i) s += sA[i];
    dst[128] = s;
  }
}

__global__ void __launch_bounds__(128) kda_bwd_param_sum_kernel(const BwdParams p) {
  const int h = blockIdx.x, c = threadIdx.x;
  // as above: sixteen partial sums over the blocks, combined in a fixed order
  float a16[16], b16[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) a16[u] = b16[u] = 0.f;
  int b = 0;
  for (; b + 16 <= p.nblk; b += 16) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float* src = p.ppart + ((size_t)(b + u) * p.H + h) * kBwdParamStride;
      a16[u] += src[c];
      if (c == 0) b16[u] += src[128];
    }
  }
  for (; b < p.nblk; ++b) {   // the tail, in order
    const float* src = p.ppart + ((size_t)b * p.H + h) * kBwdParamStride;
    a16[0] += src[c];
    if (c == 0) b16[0] += src[128];
  }
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int u = 0; u < w; ++u) {
      a16[u] += a16[u + w];
      b16[u] += b16[u + w];
    }
  const float acc = a16[0], accA = b16[0];
  if (p.ddt_bias != nullptr) p.ddt_bias[h * 128 + c] = acc;
  if (c == 0 && p.dA_log != nullptr) p.dA_log[h] = accA;
}


// ============================================================================ chunked path
// The gradient through the 16-token chunked form of the forward, differentiated chunk by
// chunk.  The backward chains (kda_chain_bwd.cu) store, per chunk, the state S0 entering it
// and the gradient dS1 of the state at its end (bf16), with Vn and dVn (fp32).  Per chunk:
//   dP  = tril(scale dO Vn^T)       dQp = scale dO S0^T + dP Km       dKm = dP^T Qp + dR^T Kp
//   dT  = dVn V^T - dVn S0^T Kp^T   dV  = Tm^T dVn                    dKp = -Tm^T dVn S0^T + dR Km
//   dA  = strict_lower(-M^T (dT Diag(beta)) M^T),  dR = Diag(beta) dA
//   dbeta_s = sum_r dT[r][s] M[r][s] + sum_s' dA[s][s'] R[s][s']
//   dG  = dKp Kp - dKm Km + dQp Qp - dKd Kd, and at the chunk's last token also
//         sum_r dKd_r Kd_r + Gam_C sum_v dS1 S0   (dKd = Vn dS1^T)
// with G the within-chunk cumsum of ghat, Gam = exp(G), Kp = kh Gam, Km = kh / Gam, Qp = qh Gam,
// Kd = kh Gam_C / Gam, R = Kp Km^T, M = (I + Diag(beta) strict_lower(R))^-1, Tm = M Diag(beta).
// Products of Gam and 1 / Gam are taken about the anchor a = G_C / 2 (exp(G - a), exp(a - G)),
// so no factor leaves exp(|G_C| / 2); the gate with a lower bound keeps |G_C| <= 80.  The chunk
// kernel keeps G in base 2 (G log2 e) and takes every factor as a power of two.
// Then dghat = reverse cumsum of dG, and the norms, the beta sigmoid and the gate as in finish.

constexpr int kXPad = 136;   // bf16 pitch of the state-product kernel's staged rows (272 bytes)
constexpr int kVPad = 132;   // bf16 pitch of the chunk kernel's v and dO rows
constexpr int kGPad = 132;   // fp32 pitch of the chunk kernel's [16][128] arrays

struct ChunkLoc {
  int64_t row;   // first token row of the chunk
  int nv;        // tokens of the chunk inside its sequence
};

// The chunk stored in slot `slot`: sequence n owns the slots n + row0(n) / 16 .. + chunks(n) - 1.
// Slots between two sequences' ranges hold no chunk (false).
__device__ __forceinline__ bool chunk_of_slot(const BwdParams& p, int64_t slot, ChunkLoc& cl) {
  if (p.N <= 0) return false;
  auto start = [&](int n) -> int64_t {
    const int64_t r0 = p.cu == nullptr ? (int64_t)n * p.T : min(max(p.cu[n], (int64_t)0), p.BT);
    return (int64_t)n + (r0 >> 4);
  };
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start(mid) <= slot) lo = mid; else hi = mid - 1;
  }
  const SeqRange sr = seq_range(p, lo, false);
  const int64_t c = slot - ((int64_t)lo + (sr.t0 >> 4));
  if (c < 0 || c * 16 >= sr.len) return false;
  cl.row = sr.t0 + c * 16;
  cl.nv = (int)min((int64_t)16, sr.len - c * 16);
  return true;
}

__device__ __forceinline__ WorkItem bwd_item(int64_t row0, int64_t len, int h, int mode, int n, int in_slot,
                                             int out_slot, int aux_slot) {
  WorkItem it;
  it.row0 = (int)row0;
  it.len = (int)len;
  it.head = h;
  it.mode = mode;
  it.seq = n;
  it.in_slot = in_slot;
  it.out_slot = out_slot;
  it.aux_slot = aux_slot;
  return it;
}

// The chains' runs.  A sequence of c chunks is cut into P = min(parts, c) parts at chunk
// boundaries (P = 1 when parts = 1 or c <= 1).  The first launch runs, per (sequence, head) and
// part j, the part's forward run (the first from the true initial state, the others from zero)
// and its reverse run (the last from dfinal or zero, the others from zero); these store S0 and
// Vn, or dS1 and dVn, and leave their final states in slots: forward part j < P - 1 in E_j,
// reverse part j in F_j (F_0 only when dh0 is wanted; with P = 1 the reverse run writes dh0).
// Correction launch l = 1 .. parts - 1 then runs, for each sequence with l < P, the forward
// correction of part l from the true state E_{l-1} and the reverse correction of part
// r = P - 1 - l from the true dS F_{r+1}.  Corrections take v (dout) as zero and add their
// part to what the parts' runs stored; each adds its final state to the slot its part's run
// left there (E_l, F_r), which then holds the true state at that cut, or gives dh0 with F_0
// added.  By linearity the sums are the uncut runs' values.  Slots of chain i: E_j at
// (2 parts - 1) i + j, F_j at (2 parts - 1) i + parts - 1 + j.  Unused entries are placeholders
// (len < 0).
__global__ void __launch_bounds__(256) kda_bwd_items_kernel(const BwdParams p) {
  const int64_t NH = (int64_t)p.N * p.H;
  const int P = p.parts;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < NH; i += stride) {
    const int n = (int)(i / p.H), h = (int)(i - (int64_t)n * p.H);
    const SeqRange sr = seq_range(p, n, h == 0);
    const int64_t chunks = (sr.len + 15) / 16;
    const int Pn = (int)(chunks < (int64_t)P ? (chunks > 1 ? chunks : 1) : P);
    auto part_row = [&](int j) {   // first row of part j (j = Pn: the sequence's end)
      return j >= Pn ? sr.t0 + sr.len : sr.t0 + 16 * ((chunks * j) / Pn);
    };
    const int base = (int)((2 * P - 1) * i);
    auto E = [&](int j) { return base + j; };
    auto F = [&](int j) { return base + P - 1 + j; };
    const int in_f = p.init_state != nullptr ? kInUser : kInZero;
    const int in_r = p.dfinal != nullptr ? kInUser : kInZero;
    const int dh = p.dh0 != nullptr ? kOutUser : kOutNone;
    const WorkItem none = bwd_item(0, -1, h, kModeForward, n, kInZero, kOutNone, -1);
    WorkItem* L = p.items + 2 * P * i;
    for (int j = 0; j < P; ++j) {
      if (j >= Pn) {
        L[j] = none;
        L[P + j] = none;
        continue;
      }
      const int64_t r0 = part_row(j), len = part_row(j + 1) - r0;
      L[j] = bwd_item(r0, len, h, kModeForward, n, j == 0 ? in_f : kInZero, j < Pn - 1 ? E(j) : kOutNone, -1);
      const int rout = Pn == 1 ? dh : (j > 0 ? F(j) : (dh == kOutUser ? F(0) : kOutNone));
      L[P + j] = bwd_item(r0, len, h, kModeReverse, n, j == Pn - 1 ? in_r : kInZero, rout, -1);
    }
    for (int l = 1; l < P; ++l) {
      WorkItem* C = p.citems + (int64_t)(l - 1) * 2 * NH + 2 * i;
      if (l >= Pn) {
        C[0] = none;
        C[1] = none;
        continue;
      }
      const int64_t f0 = part_row(l), r = Pn - 1 - l, q0 = part_row((int)r);
      const bool fout = l < Pn - 1;
      C[0] = bwd_item(f0, part_row(l + 1) - f0, h, kModeCorrect, n, E(l - 1), fout ? E(l) : kOutNone,
                      fout ? E(l) : -1);
      if (r > 0)
        C[1] = bwd_item(q0, part_row((int)r + 1) - q0, h, kModeReverseCorrect, n, F((int)r + 1), F((int)r),
                        F((int)r));
      else
        C[1] = bwd_item(q0, part_row(1) - q0, h, kModeReverseCorrect, n, F(1), dh, dh == kOutUser ? F(0) : -1);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.item_count = (int)(2 * P * NH);
    *p.citem_count = (int)(2 * NH);
  }
}

__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x, y);
  lo = pack_bf16x2(x - bf16lo_to_f32(hi), y - bf16hi_to_f32(hi));
}

// ---------------------------------------------------------------------------- state products
// Per (chunk, head): X1 = dO S0^T, X2 = Vn dS1^T, X3 = dVn S0^T ([16 tokens][128 channels],
// contractions over the 128 value rows) on bf16 warp MMA with fp32 accumulation (Vn and dVn
// split into bf16 hi + lo), and Z = sum over v of dS1 * S0 per channel, the diagonal of
// S0^T dS1.  Warp w owns channels 16 w .. 16 w + 15.
struct XprodSmem {
  // S0 and dS1 as stored (piece-major, [k / 8][v][k % 8]: 2 KB per eight channels), brought
  // in by one bulk copy each; eight consecutive v of a piece are 128 contiguous bytes, so the
  // transposed fragment loads below are conflict-free
  uint16_t s0[16 * 1024];
  uint16_t ds1[16 * 1024];
  uint16_t a[5][16][kXPad];   // dO, Vn hi, Vn lo, dVn hi, dVn lo: [token][v]
  uint64_t bar;               // the copies' completion (one phase per unit)
  int abort;
};

// The unit's rows of dO, Vn and dVn as the A operands (thread: token tid / 16, values
// 8 (tid % 16) .. + 7): loaded into registers first, stored to shared memory later.
struct XprodRows {
  uint4 x;
  float4 v0, v1, d0, d1;
};
__device__ __forceinline__ XprodRows xprod_load_a(const BwdParams& p, const ChunkLoc& cl, size_t sh, int h) {
  const int tid = threadIdx.x, t = tid >> 4, c = (tid & 15) * 8;
  XprodRows r;
  r.x = make_uint4(0u, 0u, 0u, 0u);
  if (t < cl.nv) r.x = *reinterpret_cast<const uint4*>(p.dout + ((cl.row + t) * p.H + h) * 128 + c);
  const float* vn = p.vn + sh * 2048 + t * 128 + c;
  const float* dvn = p.dvn + sh * 2048 + t * 128 + c;
  r.v0 = ld4(vn);
  r.v1 = ld4(vn + 4);
  r.d0 = ld4(dvn);
  r.d1 = ld4(dvn + 4);
  return r;
}
__device__ __forceinline__ void xprod_store_a(XprodSmem& sm, const XprodRows& r) {
  const int tid = threadIdx.x, t = tid >> 4, c = (tid & 15) * 8;
  *reinterpret_cast<uint4*>(&sm.a[0][t][c]) = r.x;
  uint32_t vh[4], vl[4], dh[4], dl[4];
  split2(r.v0.x, r.v0.y, vh[0], vl[0]);
  split2(r.v0.z, r.v0.w, vh[1], vl[1]);
  split2(r.v1.x, r.v1.y, vh[2], vl[2]);
  split2(r.v1.z, r.v1.w, vh[3], vl[3]);
  split2(r.d0.x, r.d0.y, dh[0], dl[0]);
  split2(r.d0.z, r.d0.w, dh[1], dl[1]);
  split2(r.d1.x, r.d1.y, dh[2], dl[2]);
  split2(r.d1.z, r.d1.w, dh[3], dl[3]);
  *reinterpret_cast<uint4*>(&sm.a[1][t][c]) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
  *reinterpret_cast<uint4*>(&sm.a[2][t][c]) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
  *reinterpret_cast<uint4*>(&sm.a[3][t][c]) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
  *reinterpret_cast<uint4*>(&sm.a[4][t][c]) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
}

// the bulk copies of a unit's S0 and dS1 (one thread)
__device__ __forceinline__ void xprod_issue(const BwdParams& p, XprodSmem& sm, size_t sh) {
  mbar_arrive_expect_tx(&sm.bar, 2 * 32768);
  bulk_load(sm.s0, p.s0 + sh * 16384, 32768, &sm.bar);
  bulk_load(sm.ds1, p.ds1 + sh * 16384, 32768, &sm.bar);
}

struct XprodAcc {
  float x1[2][4], x2[2][4], x3[2][4], z[2][4];
};

__device__ __forceinline__ void xprod_mma(const XprodSmem& sm, XprodAcc& r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = 16 * warp;
  const int rr = lane & 15, cofs = (lane >> 4) * 8;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) r.x1[nt][e] = r.x2[nt][e] = r.x3[nt][e] = r.z[nt][e] = 0.f;
  // the fragment rows of lane: value row v0 + rr, channels k0 + cofs .. + 7 (piece (k0 + cofs) / 8)
  const uint32_t s_base = smem_u32(sm.s0) + (uint32_t)((((k0 + cofs) >> 3) * 1024 + rr * 8) * 2);
  const uint32_t d_base = smem_u32(sm.ds1) + (uint32_t)((((k0 + cofs) >> 3) * 1024 + rr * 8) * 2);
#pragma unroll 2
  for (int ks = 0; ks < 8; ++ks) {
    const int v0 = 16 * ks;
    uint32_t a[5][4];
#pragma unroll
    for (int m = 0; m < 5; ++m) ldmatrix_x4(a[m], smem_u32(&sm.a[m][rr][v0 + cofs]));
    // B fragments (the state's [v][k] rows read transposed): registers 2 nt, 2 nt + 1 are n-tile
    // nt (channels k0 + 8 nt ..); the same registers in the order 0, 2, 1, 3 are the A fragment
    // of S0^T (rows = channels k0 .. k0 + 15, columns = v)
    uint32_t bs[4], bd[4];
    ldmatrix_x4_trans(bs, s_base + v0 * 16);
    ldmatrix_x4_trans(bd, d_base + v0 * 16);
    const uint32_t s0t[4] = {bs[0], bs[2], bs[1], bs[3]};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b_s[2] = {bs[2 * nt], bs[2 * nt + 1]};
      const uint32_t b_d[2] = {bd[2 * nt], bd[2 * nt + 1]};
      mma_bf16_16x8x16(r.x1[nt], a[0], b_s);
      mma_bf16_16x8x16(r.x3[nt], a[3], b_s);
      mma_bf16_16x8x16(r.x3[nt], a[4], b_s);
      mma_bf16_16x8x16(r.x2[nt], a[1], b_d);
      mma_bf16_16x8x16(r.x2[nt], a[2], b_d);
      mma_bf16_16x8x16(r.z[nt], s0t, b_d);
    }
  }
}

__device__ __forceinline__ void xprod_store(const BwdParams& p, size_t sh, const XprodAcc& r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = 16 * warp, g = lane >> 2, tq = lane & 3;
  float* xb = p.xp + sh * 6144;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int col = k0 + 8 * nt + 2 * tq;
    *reinterpret_cast<float2*>(xb + g * 128 + col) = make_float2(r.x1[nt][0], r.x1[nt][1]);
    *reinterpret_cast<float2*>(xb + (g + 8) * 128 + col) = make_float2(r.x1[nt][2], r.x1[nt][3]);
    *reinterpret_cast<float2*>(xb + 2048 + g * 128 + col) = make_float2(r.x2[nt][0], r.x2[nt][1]);
    *reinterpret_cast<float2*>(xb + 2048 + (g + 8) * 128 + col) = make_float2(r.x2[nt][2], r.x2[nt][3]);
    *reinterpret_cast<float2*>(xb + 4096 + g * 128 + col) = make_float2(r.x3[nt][0], r.x3[nt][1]);
    *reinterpret_cast<float2*>(xb + 4096 + (g + 8) * 128 + col) = make_float2(r.x3[nt][2], r.x3[nt][3]);
  }
  // the diagonal of S0^T dS1: channel k0 + g (n-tile 0, row g, column 2 tq + e) and channel
  // k0 + 8 + g (n-tile 1, row g + 8) sit in lane 4 g + g / 2, element e = g % 2
  if ((g >> 1) == tq) {
    const bool odd = g & 1;   // selects, not a runtime index: the accumulators stay in registers
    p.zs[sh * 128 + k0 + g] = odd ? r.z[0][1] : r.z[0][0];
    p.zs[sh * 128 + k0 + 8 + g] = odd ? r.z[1][3] : r.z[1][2];
  }
}

// ---------------------------------------------------------------------------- chunk gradients

// Per (chunk, head), 256 threads: thread (i = tid / 16, channels 8 (tid % 16) .. + 7) for the
// per-element steps, thread (i, j) = (tid / 16, tid % 16) for the 16 x 16 ones.
struct ChunkSmem {
  float qh[16][kGPad], kh[16][kGPad], G[16][kGPad];
  float Vn[16][kGPad], dVn[16][kGPad], X3[16][kGPad];
  float Kpa[16][kGPad], Kma[16][kGPad], Qpa[16][kGPad];   // kh exp(G - a), kh exp(a - G), qh exp(G - a)
  union {
    struct {   // v and dO rows (bf16), read by the first products only
      uint16_t vb[16][kVPad], dob[16][kVPad];
    } in;
    // then the A operands of the second products as tf32 {hi, lo} pairs: dP, dR, dP^T, dR^T,
    // Tm^T (pitch 20 pairs: the 64-bit fragment reads of rows g, columns k + tq are conflict-free)
    uint2 a[5][16][20];
  } u;
  // 16 x 16 matrices, pitch 20 (the warp-MMA fragment reads of rows g, columns k + tq are then
  // conflict-free); the first products' second halves (channels 64 .. 127) land in P2
  float R[16][20], dP[16][20], dVnV[16][20], dWKp[16][20], dT[16][20], M[16][20], Tm[16][20], dM[16][20];
  float P2[4][16][20];
  float Y[16][20], dA[16][20], dR[16][20];
  float beta[16], rq[16], rk[16], dbeta[16];
  float a[128], Ea[128], GC[128], Z[128];
};

__device__ __forceinline__ void unpack8(const uint4 w, float (&x)[8]) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    x[2 * u] = bf16lo_to_f32(a[u]);
    x[2 * u + 1] = bf16hi_to_f32(a[u]);
  }
}
// eight consecutive floats of shared memory as two 16-byte accesses (scalar accesses at the
// 32-byte stride of the lanes' channel groups would conflict eight ways)
__device__ __forceinline__ void ld8(const float* p, float (&x)[8]) {
  const float4 a = ld4(p), b = ld4(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void st8(float* p, const float (&x)[8]) {
  st4(p, make_float4(x[0], x[1], x[2], x[3]));
  st4(p + 4, make_float4(x[4], x[5], x[6], x[7]));
}
__device__ __forceinline__ float sum16(float x) {   // over the 16 lanes of a half-warp
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// fp32-accurate products on tf32 warp MMA: x = hi + lo with both parts tf32 (relative 2^-22),
// and A B = Ah Bh + Ah Bl + Al Bh (the Al Bl term is below fp32 rounding)
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  hi = f32_to_tf32(x);
  lo = f32_to_tf32(x - __uint_as_float(hi));
}
struct Frag4 {   // an A fragment (16 x 8) as hi and lo parts
  uint32_t h[4], l[4];
};
struct Frag2 {   // a B fragment (8 x 8)
  uint32_t h[2], l[2];
};
__device__ __forceinline__ Frag4 split4(float a0, float a1, float a2, float a3) {
  Frag4 f;
  tf32_split(a0, f.h[0], f.l[0]);
  tf32_split(a1, f.h[1], f.l[1]);
  tf32_split(a2, f.h[2], f.l[2]);
  tf32_split(a3, f.h[3], f.l[3]);
  return f;
}
__device__ __forceinline__ Frag2 split2f(float b0, float b1) {
  Frag2 f;
  tf32_split(b0, f.h[0], f.l[0]);
  tf32_split(b1, f.h[1], f.l[1]);
  return f;
}
__device__ __forceinline__ void mma3x(float (&d)[4], const Frag4& a, const Frag2& b) {
  mma_tf32_16x8x8(d, a.l, b.h);
  mma_tf32_16x8x8(d, a.h, b.l);
  mma_tf32_16x8x8(d, a.h, b.h);
}

// the hardware base-2 exponential (relative error about 2^-22) and reciprocal
__device__ __forceinline__ float sigm_fast(float x) { return rcp_approx(1.f + ex2_approx(-1.4426950408889634f * x)); }

__device__ __forceinline__ void chunk_unit(const BwdParams& p, int64_t unit) {
  const int64_t slot = unit / p.H;
  const int h = (int)(unit - slot * p.H);
  ChunkLoc cl;
  if (!chunk_of_slot(p, slot, cl)) {   // a slot without a chunk adds nothing to the parameter sums
    if (threadIdx.x <= 128) p.ppart[unit * kBwdParamStride + threadIdx.x] = 0.f;
    return;
  }
  extern __shared__ __align__(16) uint8_t csm_raw[];
  ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(csm_raw);
  const int tid = threadIdx.x;
  const int ti = tid >> 4, c0 = (tid & 15) * 8;
  const bool tv = ti < cl.nv;
  const int64_t th = (cl.row + ti) * p.H + h;
  const size_t sh = (size_t)slot * p.H + h;
  const bool norm = !(p.flags & kNoQkL2Norm), beta_pre = p.flags & kBetaPreactivated;
  const float rate = expf(p.A_log[h]);
  const float lb = p.lower_bound;
  float dtb[8];
  {
    const float4 d0 = ld4(p.dt_bias + (size_t)h * 128 + c0), d1 = ld4(p.dt_bias + (size_t)h * 128 + c0 + 4);
    dtb[0] = d0.x; dtb[1] = d0.y; dtb[2] = d0.z; dtb[3] = d0.w;
    dtb[4] = d1.x; dtb[5] = d1.y; dtb[6] = d1.z; dtb[7] = d1.w;
  }
  // ---- per element: norms, gate; staged rows
  {
    uint4 wq = make_uint4(0u, 0u, 0u, 0u), wk = wq, wg = wq, wv = wq, wo = wq;
    if (tv) {
      wq = *reinterpret_cast<const uint4*>(p.q + th * 128 + c0);
      wk = *reinterpret_cast<const uint4*>(p.k + th * 128 + c0);
      wg = *reinterpret_cast<const uint4*>(p.g + th * 128 + c0);
      wv = *reinterpret_cast<const uint4*>(p.v + th * 128 + c0);
      wo = *reinterpret_cast<const uint4*>(p.dout + th * 128 + c0);
    }
    *reinterpret_cast<uint2*>(&sm.u.in.vb[ti][c0]) = make_uint2(wv.x, wv.y);
    *reinterpret_cast<uint2*>(&sm.u.in.vb[ti][c0 + 4]) = make_uint2(wv.z, wv.w);
    *reinterpret_cast<uint2*>(&sm.u.in.dob[ti][c0]) = make_uint2(wo.x, wo.y);
    *reinterpret_cast<uint2*>(&sm.u.in.dob[ti][c0 + 4]) = make_uint2(wo.z, wo.w);
    float q[8], k[8], gg[8];
    unpack8(wq, q);
    unpack8(wk, k);
    unpack8(wg, gg);
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sq = fmaf(q[j], q[j], sq);
      sk = fmaf(k[j], k[j], sk);
    }
    sq = sum16(sq);
    sk = sum16(sk);
    const float rq = tv ? (norm ? 1.f / sqrtf(sq + 1e-6f) : 1.f) : 0.f;
    const float rk = tv ? (norm ? 1.f / sqrtf(sk + 1e-6f) : 1.f) : 0.f;
    float gh[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      q[j] *= rq;
      k[j] *= rk;
      // base-2 log-decay (the cumsum and every factor below are powers of two)
      gh[j] = tv ? lb * 1.4426950408889634f * sigm_fast(rate * (gg[j] + dtb[j])) : 0.f;
    }
    st8(&sm.qh[ti][c0], q);
    st8(&sm.kh[ti][c0], k);
    st8(&sm.G[ti][c0], gh);
    if ((tid & 15) == 0) {
      sm.rq[ti] = rq;
      sm.rk[ti] = rk;
      const float b = tv ? bfv(p.beta[th]) : 0.f;
      sm.beta[ti] = tv ? (beta_pre ? b : sigm_fast(b)) : 0.f;
    }
    const float* vn = p.vn + sh * 2048 + ti * 128 + c0;
    const float* dvn = p.dvn + sh * 2048 + ti * 128 + c0;
    const float* x3 = p.xp + sh * 6144 + 4096 + ti * 128 + c0;
    st4(&sm.Vn[ti][c0], ld4(vn));
    st4(&sm.Vn[ti][c0 + 4], ld4(vn + 4));
    st4(&sm.dVn[ti][c0], ld4(dvn));
    st4(&sm.dVn[ti][c0 + 4], ld4(dvn + 4));
    st4(&sm.X3[ti][c0], ld4(x3));
    st4(&sm.X3[ti][c0 + 4], ld4(x3 + 4));
    if (tid < 128) sm.Z[tid] = p.zs[sh * 128 + tid];
  }
  __syncthreads();
  // ---- within-chunk cumsum of ghat per channel; the anchor a = G_C / 2
  if (tid < 128) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc += sm.G[i][tid];
      sm.G[i][tid] = acc;
    }
    sm.GC[tid] = acc;
    sm.a[tid] = 0.5f * acc;
    sm.Ea[tid] = ex2_approx(0.5f * acc);
  }
  __syncthreads();
  {
    float Gv[8], av[8], kh[8], qh[8], kpa[8], kma[8], qpa[8];
    ld8(&sm.G[ti][c0], Gv);
    ld8(&sm.a[c0], av);
    ld8(&sm.kh[ti][c0], kh);
    ld8(&sm.qh[ti][c0], qh);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float d = Gv[j] - av[j];
      const float gp = ex2_approx(d), gm = ex2_approx(-d);
      kpa[j] = kh[j] * gp;
      kma[j] = kh[j] * gm;
      qpa[j] = qh[j] * gp;
    }
    st8(&sm.Kpa[ti][c0], kpa);
    st8(&sm.Kma[ti][c0], kma);
    st8(&sm.Qpa[ti][c0], qpa);
  }
  __syncthreads();
  // ---- 16 x 16 products over the 128 channels / value rows, on tf32 warp MMA: warps 2 p and
  //      2 p + 1 compute product p (R = Kp' Km'^T, dP = dO Vn^T, dVnV = dVn V^T, dWKp = X3 Kp^T)
  //      over channels 0 .. 63 and 64 .. 127, both column tiles (each operand is split once);
  //      fragments: rows g, g + 8 and k columns tq, tq + 4
  {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const int prod = warp >> 1, half = warp & 1;
    float acc[2][4] = {};
#pragma unroll 2
    for (int c = 64 * half; c < 64 * half + 64; c += 8) {
      const int ca = c + tq, cb = c + tq + 4;
      if (prod == 0) {
        const Frag4 fa = split4(sm.Kpa[g][ca], sm.Kpa[g + 8][ca], sm.Kpa[g][cb], sm.Kpa[g + 8][cb]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma3x(acc[nt], fa, split2f(sm.Kma[8 * nt + g][ca], sm.Kma[8 * nt + g][cb]));
      } else if (prod == 1) {   // dO is bf16: exact in tf32
        const uint32_t ah[4] = {f32_to_tf32(bfv(sm.u.in.dob[g][ca])), f32_to_tf32(bfv(sm.u.in.dob[g + 8][ca])),
                                f32_to_tf32(bfv(sm.u.in.dob[g][cb])), f32_to_tf32(bfv(sm.u.in.dob[g + 8][cb]))};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const Frag2 fb = split2f(sm.Vn[8 * nt + g][ca], sm.Vn[8 * nt + g][cb]);
          mma_tf32_16x8x8(acc[nt], ah, fb.l);
          mma_tf32_16x8x8(acc[nt], ah, fb.h);
        }
      } else if (prod == 2) {   // v is bf16: exact in tf32
        const Frag4 fa = split4(sm.dVn[g][ca], sm.dVn[g + 8][ca], sm.dVn[g][cb], sm.dVn[g + 8][cb]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint32_t bh[2] = {f32_to_tf32(bfv(sm.u.in.vb[8 * nt + g][ca])),
                                  f32_to_tf32(bfv(sm.u.in.vb[8 * nt + g][cb]))};
          mma_tf32_16x8x8(acc[nt], fa.l, bh);
          mma_tf32_16x8x8(acc[nt], fa.h, bh);
        }
      } else {
        const Frag4 fa = split4(sm.X3[g][ca], sm.X3[g + 8][ca], sm.X3[g][cb], sm.X3[g + 8][cb]);
        const float ea = sm.Ea[ca], eb = sm.Ea[cb];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          mma3x(acc[nt], fa, split2f(sm.Kpa[8 * nt + g][ca] * ea, sm.Kpa[8 * nt + g][cb] * eb));
      }
    }
    float (*dst)[20] = half ? sm.P2[prod] : prod == 0 ? sm.R : prod == 1 ? sm.dP : prod == 2 ? sm.dVnV : sm.dWKp;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int jc = 8 * nt + 2 * tq;
      dst[g][jc] = acc[nt][0];
      dst[g][jc + 1] = acc[nt][1];
      dst[g + 8][jc] = acc[nt][2];
      dst[g + 8][jc + 1] = acc[nt][3];
    }
  }
  __syncthreads();
  {   // the two halves added; dT = dVn V^T + dW Kp^T with dW = -X3; dP = scale dO Vn^T on and
      // below the diagonal, and dP, dP^T as tf32 pairs (v and dO are read no more)
    const int i = tid >> 4, j = tid & 15;
    sm.R[i][j] += sm.P2[0][i][j];
    sm.dT[i][j] = (sm.dVnV[i][j] + sm.P2[2][i][j]) - (sm.dWKp[i][j] + sm.P2[3][i][j]);
    const float dp = j <= i ? p.scale * (sm.dP[i][j] + sm.P2[1][i][j]) : 0.f;
    uint2 hl;
    tf32_split(dp, hl.x, hl.y);
    sm.u.a[0][i][j] = hl;
    sm.u.a[2][j][i] = hl;
  }
  __syncthreads();
  // ---- M = (I + Diag(beta) strict_lower(R))^-1, one column per thread (forward substitution)
  if (tid < 16) {
    const int j = tid;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const float bi = sm.beta[i];
      float acc = x[i];
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(-bi * sm.R[i][m], x[m], acc);
      x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sm.M[i][j] = x[i];
  }
  __syncthreads();
  {
    const int i = tid >> 4, j = tid & 15;
    const float tm = sm.M[i][j] * sm.beta[j];
    sm.Tm[i][j] = tm;
    uint2 hl;
    tf32_split(tm, hl.x, hl.y);
    sm.u.a[4][j][i] = hl;
    sm.dM[i][j] = sm.dT[i][j] * sm.beta[j];
  }
  __syncthreads();
  {   // Y = dM M^T
    const int i = tid >> 4, j = tid & 15;
    float y = 0.f;
#pragma unroll
    for (int s = 0; s < 16; ++s) y = fmaf(sm.dM[i][s], sm.M[j][s], y);
    sm.Y[i][j] = y;
  }
  __syncthreads();
  {   // dA = strict_lower(-M^T Y), dR = Diag(beta) dA
    const int i = tid >> 4, j = tid & 15;
    float d = 0.f;
    if (j < i) {
#pragma unroll
      for (int r = 0; r < 16; ++r) d = fmaf(-sm.M[r][i], sm.Y[r][j], d);
    }
    sm.dA[i][j] = d;
    sm.dR[i][j] = sm.beta[i] * d;
    uint2 hl;
    tf32_split(sm.beta[i] * d, hl.x, hl.y);
    sm.u.a[1][i][j] = hl;
    sm.u.a[3][j][i] = hl;
  }
  __syncthreads();
  if (tid < 16) {
    const int s = tid;
    float db = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) db = fmaf(sm.dT[r][s], sm.M[r][s], db);
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) db = fmaf(sm.dA[s][s2], sm.R[s][s2], db);
    sm.dbeta[s] = db;
  }
  __syncthreads();
  // ---- [16 tokens] x [128 channels] products over the chunk's tokens, on tf32 warp MMA; warp w
  //      owns channels 16 w .. + 15 (n-tiles nt = 0, 1):
  //        sq = dP Km',  sp = dR Km',  smk = dP^T Qp' + dR^T Kp',  tw = Tm^T X3,  dv = Tm^T dVn
  //      then, per element it holds (tokens g, g + 8; channels 16 w + 8 nt + 2 tq, + 1):
  //      dqh, dkh, dv, dG (before the cumsum) and dKd Kd
  {
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
    const float* xb = p.xp + sh * 6144;
#pragma unroll 1
    for (int nt = 0; nt < 2; ++nt) {
      // this n-tile's X1 and X2 elements, loaded before its MMAs so that their latency is hidden
      const int c = 16 * warp + 8 * nt + 2 * tq;
      float2 x1v[2], x2v[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        x1v[hr] = *reinterpret_cast<const float2*>(xb + (g + 8 * hr) * 128 + c);
        x2v[hr] = *reinterpret_cast<const float2*>(xb + 2048 + (g + 8 * hr) * 128 + c);
      }
      float sq[4] = {}, sp[4] = {}, smk[4] = {}, tw[4] = {}, dv[4] = {};
#pragma unroll
      for (int kk = 0; kk < 16; kk += 8) {
        const int ka = kk + tq, kb = kk + tq + 4;
        auto frag = [&](int m) {
          const uint2 a0 = sm.u.a[m][g][ka], a1 = sm.u.a[m][g + 8][ka];
          const uint2 a2 = sm.u.a[m][g][kb], a3 = sm.u.a[m][g + 8][kb];
          Frag4 f;
          f.h[0] = a0.x; f.h[1] = a1.x; f.h[2] = a2.x; f.h[3] = a3.x;
          f.l[0] = a0.y; f.l[1] = a1.y; f.l[2] = a2.y; f.l[3] = a3.y;
          return f;
        };
        const int cb = 16 * warp + 8 * nt + g;
        const Frag2 bKm = split2f(sm.Kma[ka][cb], sm.Kma[kb][cb]);
        const Frag2 bQp = split2f(sm.Qpa[ka][cb], sm.Qpa[kb][cb]);
        const Frag2 bKp = split2f(sm.Kpa[ka][cb], sm.Kpa[kb][cb]);
        const Frag2 bX3 = split2f(sm.X3[ka][cb], sm.X3[kb][cb]);
        const Frag2 bdV = split2f(sm.dVn[ka][cb], sm.dVn[kb][cb]);
        {
          const Frag4 fP = frag(0);
          mma3x(sq, fP, bKm);
        }
        {
          const Frag4 fR = frag(1);
          mma3x(sp, fR, bKm);
        }
        {
          const Frag4 fPt = frag(2);
          mma3x(smk, fPt, bQp);
        }
        {
          const Frag4 fRt = frag(3);
          mma3x(smk, fRt, bKp);
        }
        {
          const Frag4 fTt = frag(4);
          mma3x(tw, fTt, bX3);
          mma3x(dv, fTt, bdV);
        }
      }
      __syncwarp();   // every lane has read columns 16 w + 8 nt .. + 7 of Kpa, Qpa and X3: rewritten below
      const float2 av = *reinterpret_cast<const float2*>(&sm.a[c]);
      const float2 eav = *reinterpret_cast<const float2*>(&sm.Ea[c]);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = g + 8 * hr;
        const float2 Gv = *reinterpret_cast<const float2*>(&sm.G[i][c]);
        const float2 khv = *reinterpret_cast<const float2*>(&sm.kh[i][c]);
        const float2 qhv = *reinterpret_cast<const float2*>(&sm.qh[i][c]);
        const float2 x1 = x1v[hr], x2 = x2v[hr];
        const float Ge[2] = {Gv.x, Gv.y}, ae[2] = {av.x, av.y}, eae[2] = {eav.x, eav.y};
        const float khe[2] = {khv.x, khv.y}, qhe[2] = {qhv.x, qhv.y}, x1e[2] = {x1.x, x1.y}, x2e[2] = {x2.x, x2.y};
        float dqh[2], dkh[2], dG[2], dkdkh[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 2 * hr + e;   // accumulator element: (row g + 8 hr, column 2 tq + e)
          // with the anchor a = G_C / 2: 2^G = 2^(G - a) 2^a and 2^(G_C - G) = 2^(a - G) 2^a
          const float d = Ge[e] - ae[e];
          const float gp = ex2_approx(d), gm = ex2_approx(-d);
          const float gam = gp * eae[e], dk = gm * eae[e];
          dqh[e] = p.scale * x1e[e] * gam + gp * sq[r];
          const float dkp = -tw[r] * gam + gp * sp[r];
          const float dkm = gm * smk[r];
          const float dkd = x2e[e] * dk;
          dkh[e] = dkp + dkm + dkd;
          dG[e] = (dkp - dkm - dkd) * khe[e] + dqh[e] * qhe[e];
          dkdkh[e] = dkd * khe[e];
        }
        *reinterpret_cast<float2*>(&sm.Kpa[i][c]) = make_float2(dqh[0], dqh[1]);
        *reinterpret_cast<float2*>(&sm.Qpa[i][c]) = make_float2(dkh[0], dkh[1]);
        *reinterpret_cast<float2*>(&sm.Vn[i][c]) = make_float2(dG[0], dG[1]);
        *reinterpret_cast<float2*>(&sm.X3[i][c]) = make_float2(dkdkh[0], dkdkh[1]);
        if (i < cl.nv) {
          const int64_t thi = (cl.row + i) * p.H + h;
          *reinterpret_cast<float2*>(p.dv + thi * 128 + c) = make_float2(dv[2 * hr], dv[2 * hr + 1]);
        }
      }
    }
  }
  __syncthreads();
  // g of this thread's token and channels, for the gate's chain rule at the end (loaded now, so
  // that its latency passes during the per-channel step)
  uint4 wg = make_uint4(0u, 0u, 0u, 0u);
  if (tv) wg = *reinterpret_cast<const uint4*>(p.g + th * 128 + c0);
  // ---- per channel: the last token's terms, then the reverse cumsum (dghat)
  if (tid < 128) {
    const int c = tid, last = cl.nv - 1;
    float sl = ex2_approx(sm.GC[c]) * sm.Z[c];
    for (int i = 0; i <= last; ++i) sl += sm.X3[i][c];
    float acc = 0.f;
    for (int i = last; i >= 0; --i) {
      acc += sm.Vn[i][c] + (i == last ? sl : 0.f);
      sm.Vn[i][c] = acc;
    }
  }
  __syncthreads();
  // ---- per token: the norms, the beta sigmoid and the gate
  {
    float qh[8], kh[8], dgh[8], dqh[8], dkh[8];
    ld8(&sm.qh[ti][c0], qh);
    ld8(&sm.kh[ti][c0], kh);
    ld8(&sm.Vn[ti][c0], dgh);
    ld8(&sm.Kpa[ti][c0], dqh);
    ld8(&sm.Qpa[ti][c0], dkh);
    float qd = 0.f, kd = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qd = fmaf(qh[j], dqh[j], qd);
      kd = fmaf(kh[j], dkh[j], kd);
    }
    qd = sum16(qd);
    kd = sum16(kd);
    const float rq = sm.rq[ti], rk = sm.rk[ti];
    float dq[8], dk[8], dg[8], wa = 0.f;
    float gg[8];
    unpack8(wg, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dq[j] = norm ? rq * (dqh[j] - qh[j] * qd) : dqh[j];
      dk[j] = norm ? rk * (dkh[j] - kh[j] * kd) : dkh[j];
      // ghat = lb sigmoid(z), z = rate x: d/dx = rate lb s (1 - s); d/dA_log = x d/dx
      const float x = gg[j] + dtb[j], sg = sigm_fast(rate * x);
      dg[j] = dgh[j] * lb * sg * (1.f - sg) * rate;
      wa = fmaf(dg[j], x, wa);
    }
    wa = sum16(wa);
    if (tv) {
      st4(p.dq + th * 128 + c0, make_float4(dq[0], dq[1], dq[2], dq[3]));
      st4(p.dq + th * 128 + c0 + 4, make_float4(dq[4], dq[5], dq[6], dq[7]));
      st4(p.dk + th * 128 + c0, make_float4(dk[0], dk[1], dk[2], dk[3]));
      st4(p.dk + th * 128 + c0 + 4, make_float4(dk[4], dk[5], dk[6], dk[7]));
      st4(p.dg + th * 128 + c0, make_float4(dg[0], dg[1], dg[2], dg[3]));
      st4(p.dg + th * 128 + c0 + 4, make_float4(dg[4], dg[5], dg[6], dg[7]));
      if ((tid & 15) == 0) {
        const float b = sm.beta[ti];
        p.dbeta[th] = beta_pre ? sm.dbeta[ti] : sm.dbeta[ti] * b * (1.f - b);
      }
    }
    // this unit's parameter partials: d dt_bias summed over the chunk's tokens (per channel) and
    // the dA_log terms summed; the units are summed in a fixed order afterwards
    __syncthreads();   // Kma and Y are read no more
#pragma unroll
    for (int j = 0; j < 8; ++j) dg[j] = tv ? dg[j] : 0.f;
    st8(&sm.Kma[ti][c0], dg);
    if ((tid & 15) == 0) sm.Y[0][ti] = tv ? wa : 0.f;
    __syncthreads();
    if (tid < 128) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc += sm.Kma[i][tid];
      p.ppart[unit * kBwdParamStride + tid] = acc;
    } else if (tid == 128) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc += sm.Y[0][i];
      p.ppart[unit * kBwdParamStride + 128] = acc;
    }
  }
}

// Grid (ceil(nslots / 64), H): block b sums the partials of the 64 units (slots 64 b .. 64 b + 63,
// head h) in slot order, sixteen loads in flight; kda_bwd_param_sum_kernel then sums the blocks.
__global__ void __launch_bounds__(128) kda_bwd_unit_sum_kernel(const BwdParams p, float* out) {
  const int blk = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int64_t s0 = (int64_t)blk * 64, s1 = min(p.nslots, s0 + 64);
  float a16[16], b16[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) a16[u] = b16[u] = 0.f;
  int64_t sl = s0;
  for (; sl + 16 <= s1; sl += 16) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float* src = p.ppart + ((sl + u) * p.H + h) * kBwdParamStride;
      a16[u] += src[c];
      if (c == 0) b16[u] += src[128];
    }
  }
  for (; sl < s1; ++sl) {   // the tail, in order
    const float* src = p.ppart + (sl * p.H + h) * kBwdParamStride;
    a16[0] += src[c];
    if (c == 0) b16[0] += src[128];
  }
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int u = 0; u < w; ++u) {
      a16[u] += a16[u + w];
      b16[u] += b16[u + w];
    }
  float* dst = out + ((size_t)blk * p.H + h) * kBwdParamStride;
  dst[c] = a16[0];
  if (c == 0) dst[128] = b16[0];
}

// Persistent CTAs (two per SM) walk the units, heads fastest (the CTAs working at once read
// every head of a few chunks, so each token row is read whole from DRAM).  The next unit's S0
// and dS1 copies are requested as soon as this unit's products have read the buffers, and its
// A operands staged while they arrive; the wait on them is bounded (timeout: the error word's
// timeout bit, and the CTA stops after its copies in flight have landed).
__global__ void __launch_bounds__(256, 2) kda_bwd_xprod_kernel(const BwdParams p) {
  extern __shared__ __align__(128) uint8_t xsm_raw[];
  XprodSmem& sm = *reinterpret_cast<XprodSmem*>(xsm_raw);
  const int64_t units = p.nslots * p.H;
  const int tid = threadIdx.x;
  auto locate = [&](int64_t u, ChunkLoc& cl, size_t& sh, int& h) {
    const int64_t slot = u / p.H;
    h = (int)(u - slot * p.H);
    sh = (size_t)slot * p.H + h;
    return u < units && chunk_of_slot(p, slot, cl);
  };
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const AbortState ab{&sm.abort, p.err};
  int64_t u = blockIdx.x;
  ChunkLoc cl;
  size_t sh;
  int h;
  bool valid = locate(u, cl, sh, h);
  if (valid) {
    if (tid == 0) xprod_issue(p, sm, sh);
    xprod_store_a(sm, xprod_load_a(p, cl, sh, h));
  }
  __syncthreads();
  uint32_t phase = 0;
  bool pending = valid;   // a copy of this CTA is in flight
  for (; u < units; u += gridDim.x) {
    XprodAcc r;
    if (valid) {
      const bool ok = mbar_wait(&sm.bar, phase, ab);
      if (ok) {
        phase ^= 1u;   // a copy that did not land keeps its phase for the drain below
        pending = false;
        xprod_mma(sm, r);
      }
    }
    __syncthreads();   // every warp is done with the buffers (or the CTA is stopping)
    if (sm.abort) break;
    ChunkLoc ncl;
    size_t nsh;
    int nh;
    const bool nvalid = locate(u + gridDim.x, ncl, nsh, nh);
    if (nvalid && tid == 0) {
      fence_proxy_async_smem();
      xprod_issue(p, sm, nsh);
    }
    pending = pending || nvalid;
    // the next unit's rows are requested before this unit's products are written out
    XprodRows rows;
    if (nvalid) rows = xprod_load_a(p, ncl, nsh, nh);
    if (valid) xprod_store(p, sh, r);
    if (nvalid) xprod_store_a(sm, rows);
    __syncthreads();
    valid = nvalid;
    cl = ncl;
    sh = nsh;
    h = nh;
  }
  if (pending) mbar_wait_drain(&sm.bar, phase);
}
__global__ void __launch_bounds__(256, 2) kda_bwd_chunk_kernel(const BwdParams p) {
  const int64_t units = p.nslots * p.H;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    chunk_unit(p, u);
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, int phase, cudaStream_t s) {
  const int64_t TH = p.BT * p.H;
  const int warp_grid = (int)std::min<int64_t>((TH + 3) / 4, 152 * 32);
  const int64_t rec_grid = (int64_t)p.N * p.H * kBwdSlices;
  cudaError_t e = cudaSuccess;
  switch (phase) {
    case 0:   // error word, per token-head vectors
      if ((e = cudaMemsetAsync(p.err, 0, sizeof(int), s)) != cudaSuccess) return e;
      if (TH > 0) kda_bwd_prep_kernel<<<warp_grid, 128, 0, s>>>(p);
      return cudaGetLastError();
    case 1:   // forward recurrence with stored states
      if (rec_grid > 0) kda_bwd_ckpt_kernel<<<(unsigned)rec_grid, kThreads, 0, s>>>(p);
      return cudaGetLastError();
    case 2:   // reverse recurrence
      if (rec_grid > 0) kda_bwd_reverse_kernel<<<(unsigned)rec_grid, kThreads, 0, s>>>(p);
      return cudaGetLastError();
    case 3: {  // chain rule per token-head, parameter sums
      if (TH > 0) {
        kda_bwd_finish_kernel<<<warp_grid, 128, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      const bool params = !(p.flags & kGatePreactivated) && (p.dA_log != nullptr || p.ddt_bias != nullptr);
      if (params) {
        if (p.nblk > 0) {
          kda_bwd_param_kernel<<<dim3(p.nblk, p.H), 128, 0, s>>>(p);
          if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        kda_bwd_param_sum_kernel<<<p.H, 128, 0, s>>>(p);
        return cudaGetLastError();
      }
      // a pre-activated gate has no parameters: their gradients are zero
      if (p.dA_log != nullptr && (e = cudaMemsetAsync(p.dA_log, 0, sizeof(float) * p.H, s)) != cudaSuccess)
        return e;
      if (p.ddt_bias != nullptr) e = cudaMemsetAsync(p.ddt_bias, 0, sizeof(float) * 128 * p.H, s);
      return e;
    }
  }
  return cudaErrorInvalidValue;
}


cudaError_t launch_bwd_chunked(const BwdParams& p, int phase, cudaStream_t s) {
  // the dynamic shared-memory opt-in is a per-device setting: made once per device
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    if ((e = cudaFuncSetAttribute(kda_bwd_xprod_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sizeof(XprodSmem))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(kda_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sizeof(ChunkSmem))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  const int64_t NH = (int64_t)p.N * p.H;
  const unsigned slots_grid = (unsigned)std::max<int64_t>(std::min<int64_t>(p.nslots * p.H, 2 * (int64_t)p.sms), 1);
  switch (phase) {
    case 0: {   // error word, the chains' runs
      if ((e = cudaMemsetAsync(p.err, 0, sizeof(int), s)) != cudaSuccess) return e;
      const int grid = (int)std::min<int64_t>(std::max<int64_t>((NH + 255) / 256, 1), 1024);
      kda_bwd_items_kernel<<<grid, 256, 0, s>>>(p);
      return cudaGetLastError();
    }
    case 2:   // state products
      if (p.nslots > 0 && p.BT > 0) kda_bwd_xprod_kernel<<<slots_grid, 256, sizeof(XprodSmem), s>>>(p);
      return cudaGetLastError();
    case 3: {  // chunk gradients, parameter sums
      if (p.nslots > 0 && p.BT > 0) {
        kda_bwd_chunk_kernel<<<slots_grid, 256, sizeof(ChunkSmem), s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      if (p.dA_log != nullptr || p.ddt_bias != nullptr) {
        // the units' partials, summed in slot blocks of 64, then over the blocks
        const int nb = (int)((p.nslots + 63) / 64);
        float* blocks = p.ppart + (size_t)std::max<int64_t>(p.nslots, 1) * p.H * kBwdParamStride;
        if (nb > 0) {
          kda_bwd_unit_sum_kernel<<<dim3(nb, p.H), 128, 0, s>>>(p, blocks);
          if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        BwdParams q = p;
        q.ppart = blocks;
        q.nblk = nb;
        kda_bwd_param_sum_kernel<<<p.H, 128, 0, s>>>(q);
      }
      return cudaGetLastError();
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
