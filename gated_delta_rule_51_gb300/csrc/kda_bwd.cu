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
// Kernels, in launch order:
//   prep     per token-head: alpha = exp(ghat), beta, qh, kh and the norms' scales;
//   ckpt     the forward recurrence, storing the state at every kBwdChunk-th token;
//   reverse  per chunk, last first: for each token (last first) the state before it is
//            recomputed from the chunk's stored state (or from the state before the
//            chunk's middle token, kept once per chunk), then the reverse step runs; the
//            per-token column partials of dqh, dkh, dalpha, dbeta go to the workspace;
//   finish   per token-head: the partials summed, then the norms, the sigmoid and the gate;
//   param    dA_log and dt_bias summed over tokens in blocks, then over blocks.
// Memory: the stored states take (B T / kBwdChunk + N + 1) x H x 64 KiB.  No kernel waits
// on another CTA; the only barriers are __syncthreads.
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
  float acc = 0.f, accA = 0.f;
  for (int64_t t = t0; t < t1; ++t) acc += p.dg[(t * p.H + h) * 128 + c];
  for (int64_t t = t0 + c; t < t1; t += 128) accA += p.dA_tok[t * p.H + h];
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
  float acc = 0.f, accA = 0.f;
  for (int b = 0; b < p.nblk; ++b) {
    const float* src = p.ppart + ((size_t)b * p.H + h) * kBwdParamStride;
    acc += src[c];
    if (c == 0) accA += src[128];
  }
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
// so no factor leaves exp(|G_C| / 2); the gate with a lower bound keeps |G_C| <= 80.
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

// The chains' runs: per (sequence, head) a forward run storing S0 and Vn, then the same count
// of reverse runs carrying dS from dfinal (or zero) to dh0.
__global__ void __launch_bounds__(256) kda_bwd_items_kernel(const BwdParams p) {
  const int64_t NH = (int64_t)p.N * p.H;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * NH; i += stride) {
    const bool rev = i >= NH;
    const int64_t r = rev ? i - NH : i;
    const int n = (int)(r / p.H), h = (int)(r - (int64_t)n * p.H);
    const SeqRange sr = seq_range(p, n, !rev && h == 0);
    WorkItem it;
    it.row0 = (int)sr.t0;
    it.len = (int)sr.len;
    it.head = h;
    it.mode = rev ? kModeReverse : kModeForward;
    it.seq = n;
    it.in_slot = (rev ? p.dfinal != nullptr : p.init_state != nullptr) ? kInUser : kInZero;
    it.out_slot = (rev && p.dh0 != nullptr) ? kOutUser : kOutNone;
    it.aux_slot = -1;
    p.items[i] = it;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.item_count = (int)(2 * NH);
}

__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x, y);
  lo = pack_bf16x2(x - bf16lo_to_f32(hi), y - bf16hi_to_f32(hi));
}

// ---------------------------------------------------------------------------- state products
// Per (chunk, head): X1 = dO S0^T, X2 = Vn dS1^T, X3 = dVn S0^T ([16 tokens][128 channels],
// contractions over the 128 value rows) on bf16 warp MMA with fp32 accumulation (Vn and dVn
// split into bf16 hi + lo), and Z = sum over v of dS1 * S0 per channel.  Warp w owns channels
// 16 w .. 16 w + 15.
struct XprodSmem {
  uint16_t s0[128][kXPad];    // [v][k]
  uint16_t ds1[128][kXPad];
  uint16_t a[5][16][kXPad];   // dO, Vn hi, Vn lo, dVn hi, dVn lo: [token][v]
  float z[2][128];
};

__global__ void __launch_bounds__(256, 2) kda_bwd_xprod_kernel(const BwdParams p) {
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  ChunkLoc cl;
  if (!chunk_of_slot(p, slot, cl)) return;
  extern __shared__ __align__(16) uint8_t xsm_raw[];
  XprodSmem& sm = *reinterpret_cast<XprodSmem*>(xsm_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t sh = (size_t)slot * p.H + h;
  {
    const uint4* a = reinterpret_cast<const uint4*>(p.s0 + sh * 16384);
    const uint4* b = reinterpret_cast<const uint4*>(p.ds1 + sh * 16384);
    for (int i = tid; i < 2048; i += 256) {
      const int v = i >> 4, c = (i & 15) * 8;
      *reinterpret_cast<uint4*>(&sm.s0[v][c]) = a[i];
      *reinterpret_cast<uint4*>(&sm.ds1[v][c]) = b[i];
    }
  }
  {
    const int t = tid >> 4, c = (tid & 15) * 8;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (t < cl.nv) x = *reinterpret_cast<const uint4*>(p.dout + ((cl.row + t) * p.H + h) * 128 + c);
    *reinterpret_cast<uint4*>(&sm.a[0][t][c]) = x;
    const float* vn = p.vn + sh * 2048 + t * 128 + c;
    const float* dvn = p.dvn + sh * 2048 + t * 128 + c;
    const float4 v0 = ld4(vn), v1 = ld4(vn + 4), d0 = ld4(dvn), d1 = ld4(dvn + 4);
    uint32_t vh[4], vl[4], dh[4], dl[4];
    split2(v0.x, v0.y, vh[0], vl[0]);
    split2(v0.z, v0.w, vh[1], vl[1]);
    split2(v1.x, v1.y, vh[2], vl[2]);
    split2(v1.z, v1.w, vh[3], vl[3]);
    split2(d0.x, d0.y, dh[0], dl[0]);
    split2(d0.z, d0.w, dh[1], dl[1]);
    split2(d1.x, d1.y, dh[2], dl[2]);
    split2(d1.z, d1.w, dh[3], dl[3]);
    *reinterpret_cast<uint4*>(&sm.a[1][t][c]) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
    *reinterpret_cast<uint4*>(&sm.a[2][t][c]) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
    *reinterpret_cast<uint4*>(&sm.a[3][t][c]) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
    *reinterpret_cast<uint4*>(&sm.a[4][t][c]) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
  }
  __syncthreads();
  // fragments: A rows = tokens (ldmatrix row r of matrix lane >> 3), B = the state's [v][k]
  // rows read transposed (column-major 16 v x 8 k per n-tile)
  const int k0 = 16 * warp;
  const int r = lane & 15, cofs = (lane >> 4) * 8;
  float x1[2][4] = {}, x2[2][4] = {}, x3[2][4] = {};
#pragma unroll 2
  for (int ks = 0; ks < 8; ++ks) {
    const int v0 = 16 * ks;
    uint32_t a[5][4];
#pragma unroll
    for (int m = 0; m < 5; ++m) ldmatrix_x4(a[m], smem_u32(&sm.a[m][r][v0 + cofs]));
    uint32_t bs[4], bd[4];
    ldmatrix_x4_trans(bs, smem_u32(&sm.s0[v0 + r][k0 + cofs]));
    ldmatrix_x4_trans(bd, smem_u32(&sm.ds1[v0 + r][k0 + cofs]));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b_s[2] = {bs[2 * nt], bs[2 * nt + 1]};
      const uint32_t b_d[2] = {bd[2 * nt], bd[2 * nt + 1]};
      mma_bf16_16x8x16(x1[nt], a[0], b_s);
      mma_bf16_16x8x16(x3[nt], a[3], b_s);
      mma_bf16_16x8x16(x3[nt], a[4], b_s);
      mma_bf16_16x8x16(x2[nt], a[1], b_d);
      mma_bf16_16x8x16(x2[nt], a[2], b_d);
    }
  }
  {
    const int k = tid & 127, half = tid >> 7;
    float z = 0.f;
    for (int v = 64 * half; v < 64 * half + 64; ++v) z = fmaf(bfv(sm.s0[v][k]), bfv(sm.ds1[v][k]), z);
    sm.z[half][k] = z;
  }
  float* xb = p.xp + sh * 6144;
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int col = k0 + 8 * nt + 2 * tq;
    *reinterpret_cast<float2*>(xb + g * 128 + col) = make_float2(x1[nt][0], x1[nt][1]);
    *reinterpret_cast<float2*>(xb + (g + 8) * 128 + col) = make_float2(x1[nt][2], x1[nt][3]);
    *reinterpret_cast<float2*>(xb + 2048 + g * 128 + col) = make_float2(x2[nt][0], x2[nt][1]);
    *reinterpret_cast<float2*>(xb + 2048 + (g + 8) * 128 + col) = make_float2(x2[nt][2], x2[nt][3]);
    *reinterpret_cast<float2*>(xb + 4096 + g * 128 + col) = make_float2(x3[nt][0], x3[nt][1]);
    *reinterpret_cast<float2*>(xb + 4096 + (g + 8) * 128 + col) = make_float2(x3[nt][2], x3[nt][3]);
  }
  __syncthreads();
  if (tid < 128) p.zs[sh * 128 + tid] = sm.z[0][tid] + sm.z[1][tid];
}

// ---------------------------------------------------------------------------- chunk gradients
// Per (chunk, head), 256 threads: thread (i = tid / 16, channels 8 (tid % 16) .. + 7) for the
// per-element steps, thread (i, j) = (tid / 16, tid % 16) for the 16 x 16 ones.
struct ChunkSmem {
  float qh[16][kGPad], kh[16][kGPad], G[16][kGPad];
  float Vn[16][kGPad], dVn[16][kGPad], X3[16][kGPad];
  float Kpa[16][kGPad], Kma[16][kGPad], Qpa[16][kGPad];   // kh exp(G - a), kh exp(a - G), qh exp(G - a)
  uint16_t vb[16][kVPad], dob[16][kVPad];
  float R[16][17], dP[16][17], dT[16][17], M[16][17], Tm[16][17], dM[16][17], Y[16][17], dA[16][17], dR[16][17];
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
__device__ __forceinline__ float sum16(float x) {   // over the 16 lanes of a half-warp
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(256, 2) kda_bwd_chunk_kernel(const BwdParams p) {
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  ChunkLoc cl;
  if (!chunk_of_slot(p, slot, cl)) return;
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
    *reinterpret_cast<uint2*>(&sm.vb[ti][c0]) = make_uint2(wv.x, wv.y);
    *reinterpret_cast<uint2*>(&sm.vb[ti][c0 + 4]) = make_uint2(wv.z, wv.w);
    *reinterpret_cast<uint2*>(&sm.dob[ti][c0]) = make_uint2(wo.x, wo.y);
    *reinterpret_cast<uint2*>(&sm.dob[ti][c0 + 4]) = make_uint2(wo.z, wo.w);
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
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sm.qh[ti][c0 + j] = q[j] * rq;
      sm.kh[ti][c0 + j] = k[j] * rk;
      sm.G[ti][c0 + j] = tv ? lb * sigm(rate * (gg[j] + dtb[j])) : 0.f;
    }
    if ((tid & 15) == 0) {
      sm.rq[ti] = rq;
      sm.rk[ti] = rk;
      const float b = tv ? bfv(p.beta[th]) : 0.f;
      sm.beta[ti] = tv ? (beta_pre ? b : sigm(b)) : 0.f;
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
    sm.Ea[tid] = expf(0.5f * acc);
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = c0 + j;
    const float d = sm.G[ti][c] - sm.a[c];
    const float gp = expf(d), gm = expf(-d);
    const float kh = sm.kh[ti][c], qh = sm.qh[ti][c];
    sm.Kpa[ti][c] = kh * gp;
    sm.Kma[ti][c] = kh * gm;
    sm.Qpa[ti][c] = qh * gp;
  }
  __syncthreads();
  // ---- 16 x 16 products over 128 channels / value rows
  {
    const int i = tid >> 4, j = tid & 15;
    float r = 0.f, dp = 0.f, dvv = 0.f, dwk = 0.f;
#pragma unroll 4
    for (int c = 0; c < 128; c += 4) {
      const float4 kpi = ld4(&sm.Kpa[i][c]), kmj = ld4(&sm.Kma[j][c]), kpj = ld4(&sm.Kpa[j][c]);
      const float4 x3i = ld4(&sm.X3[i][c]), ea = ld4(&sm.Ea[c]);
      const float4 dvi = ld4(&sm.dVn[i][c]), vnj = ld4(&sm.Vn[j][c]);
      const float4 vj = bf4(&sm.vb[j][c]), oi = bf4(&sm.dob[i][c]);
      r += dot4(kpi, kmj);
      dwk += x3i.x * kpj.x * ea.x + x3i.y * kpj.y * ea.y + x3i.z * kpj.z * ea.z + x3i.w * kpj.w * ea.w;
      dvv += dot4(dvi, vj);
      dp += dot4(oi, vnj);
    }
    sm.R[i][j] = r;
    sm.dP[i][j] = j <= i ? p.scale * dp : 0.f;
    sm.dT[i][j] = dvv - dwk;   // dVn V^T + dW Kp^T with dW = -X3
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
    sm.Tm[i][j] = sm.M[i][j] * sm.beta[j];
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
  // ---- per element: dqh, dkh, dv, dG (before the cumsum) and dKd Kd
  float dqh[8], dkh[8], dG[8], dkdkh[8];
  {
    const float* xb = p.xp + sh * 6144 + ti * 128 + c0;
    float x1[8], x2[8];
    {
      const float4 a0 = ld4(xb), a1 = ld4(xb + 4), b0 = ld4(xb + 2048), b1 = ld4(xb + 2048 + 4);
      x1[0] = a0.x; x1[1] = a0.y; x1[2] = a0.z; x1[3] = a0.w; x1[4] = a1.x; x1[5] = a1.y; x1[6] = a1.z; x1[7] = a1.w;
      x2[0] = b0.x; x2[1] = b0.y; x2[2] = b0.z; x2[3] = b0.w; x2[4] = b1.x; x2[5] = b1.y; x2[6] = b1.z; x2[7] = b1.w;
    }
    float sq[8] = {}, sp[8] = {}, smk[8] = {}, tw[8] = {}, dv[8] = {};
#pragma unroll 2
    for (int j = 0; j < 16; ++j) {
      const float dpij = sm.dP[ti][j], drij = sm.dR[ti][j], dpji = sm.dP[j][ti], drji = sm.dR[j][ti];
      const float tmji = sm.Tm[j][ti];
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4) {
        const float4 km = ld4(&sm.Kma[j][c0 + h4]), qp = ld4(&sm.Qpa[j][c0 + h4]), kp = ld4(&sm.Kpa[j][c0 + h4]);
        const float4 x3 = ld4(&sm.X3[j][c0 + h4]), dn = ld4(&sm.dVn[j][c0 + h4]);
        const float kmv[4] = {km.x, km.y, km.z, km.w}, qpv[4] = {qp.x, qp.y, qp.z, qp.w};
        const float kpv[4] = {kp.x, kp.y, kp.z, kp.w}, x3v[4] = {x3.x, x3.y, x3.z, x3.w};
        const float dnv[4] = {dn.x, dn.y, dn.z, dn.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sq[h4 + u] = fmaf(dpij, kmv[u], sq[h4 + u]);
          sp[h4 + u] = fmaf(drij, kmv[u], sp[h4 + u]);
          smk[h4 + u] = fmaf(dpji, qpv[u], fmaf(drji, kpv[u], smk[h4 + u]));
          tw[h4 + u] = fmaf(tmji, x3v[u], tw[h4 + u]);
          dv[h4 + u] = fmaf(tmji, dnv[u], dv[h4 + u]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + j;
      const float Gv = sm.G[ti][c], d = Gv - sm.a[c];
      const float gam = expf(Gv), gp = expf(d), gm = expf(-d), dk = expf(sm.GC[c] - Gv);
      const float kh = sm.kh[ti][c], qh = sm.qh[ti][c];
      dqh[j] = p.scale * x1[j] * gam + gp * sq[j];
      const float dkp = -tw[j] * gam + gp * sp[j];
      const float dkm = gm * smk[j];
      const float dkd = x2[j] * dk;
      dkh[j] = dkp + dkm + dkd;
      dG[j] = (dkp - dkm - dkd) * kh + dqh[j] * qh;
      dkdkh[j] = dkd * kh;
    }
    if (tv) {
      st4(p.dv + th * 128 + c0, make_float4(dv[0], dv[1], dv[2], dv[3]));
      st4(p.dv + th * 128 + c0 + 4, make_float4(dv[4], dv[5], dv[6], dv[7]));
    }
  }
  __syncthreads();   // every read of Vn and X3 is done: they now hold dG and dKd Kd
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sm.Vn[ti][c0 + j] = dG[j];
    sm.X3[ti][c0 + j] = dkdkh[j];
  }
  __syncthreads();
  // ---- per channel: the last token's terms, then the reverse cumsum (dghat)
  if (tid < 128) {
    const int c = tid, last = cl.nv - 1;
    float sl = expf(sm.GC[c]) * sm.Z[c];
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
    float qd = 0.f, kd = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qd = fmaf(sm.qh[ti][c0 + j], dqh[j], qd);
      kd = fmaf(sm.kh[ti][c0 + j], dkh[j], kd);
    }
    qd = sum16(qd);
    kd = sum16(kd);
    const float rq = sm.rq[ti], rk = sm.rk[ti];
    float dq[8], dk[8], dg[8], wa = 0.f;
    float gg[8];
    {
      uint4 wg = make_uint4(0u, 0u, 0u, 0u);
      if (tv) wg = *reinterpret_cast<const uint4*>(p.g + th * 128 + c0);
      unpack8(wg, gg);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + j;
      dq[j] = norm ? rq * (dqh[j] - sm.qh[ti][c] * qd) : dqh[j];
      dk[j] = norm ? rk * (dkh[j] - sm.kh[ti][c] * kd) : dkh[j];
      // ghat = lb sigmoid(z), z = rate x: d/dx = rate lb s (1 - s); d/dA_log = x d/dx
      const float x = gg[j] + dtb[j], sg = sigm(rate * x);
      dg[j] = sm.Vn[ti][c] * lb * sg * (1.f - sg) * rate;
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
        p.dA_tok[th] = wa;
      }
    }
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
  const dim3 slots_grid((unsigned)std::max<int64_t>(p.nslots, 1), (unsigned)p.H);
  switch (phase) {
    case 0: {   // error word, the chains' runs
      if ((e = cudaMemsetAsync(p.err, 0, sizeof(int), s)) != cudaSuccess) return e;
      const int grid = (int)std::min<int64_t>(std::max<int64_t>((2 * NH + 255) / 256, 1), 1024);
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
        if (p.nblk > 0) {
          kda_bwd_param_kernel<<<dim3(p.nblk, p.H), 128, 0, s>>>(p);
          if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        kda_bwd_param_sum_kernel<<<p.H, 128, 0, s>>>(p);
      }
      return cudaGetLastError();
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
