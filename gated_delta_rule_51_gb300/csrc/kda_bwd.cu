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

}  // namespace kda
