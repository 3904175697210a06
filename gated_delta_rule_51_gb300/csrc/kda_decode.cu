// kda_decode.cu -- the recurrent step of KDA for decoding: a few tokens per
// sequence, the state read from and written back to HBM once per call.
//
// Per (sequence n, head h) and token t, with K = 128 (or 64) and V = 64, 128 or 256, the
// state kept as S^T (row v holds S[:, v] over the key channels k), the step is the KDA
// recurrence itself (FlashKDA README "Kernel API" parameter table for the
// inputs, gate and layout):
//   ghat  = lower_bound * sigmoid(exp(A_log[h]) * (g_t + dt_bias[h, :]))   (or g_t given, or
//           -exp(A_log[h]) * softplus(g_t + dt_bias[h, :]) for the gate without a lower bound)
//   beta  = sigmoid(beta logit) (or given);  qh, kh = x / sqrt(|x|^2 + 1e-6) (or as given)
//   row v of S^T:  s <- s * exp(ghat);  s <- s + beta (v_v - s . kh) kh
//   o_v   = scale * s . qh        (from the updated row)
// Rows are independent, so the work is bandwidth-bound: V / kDecRows CTAs per
// (n, h), each of kDecRows rows in warps of sixteen, every lane holding four key
// channels of each of its rows in registers for all the call's tokens.  The state
// is read once (V x K fp32 or bf16 per head) and written once.
#include <cuda_bf16.h>

#include <array>
#include <utility>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRowsPerWarp = 16;
constexpr int kDecRows = 64;                        // state rows per CTA (four CTAs per SM)
constexpr int kDecThreads = 2 * kDecRows;           // 16 rows a warp; at least 128 threads
constexpr int kDecK64 = 16;                          // kernel variant bit: K = 64
static_assert(kDecThreads >= 128, "the per-channel vectors take 128 threads");

__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// every lane ends with the full sums of all sixteen rows
__device__ __forceinline__ void warp_sum16(float (&x)[kRowsPerWarp]) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) x[r] += __shfl_xor_sync(0xffffffffu, x[r], m);
}

__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + expf(-x)); }
// log(1 + exp(x)) without overflow
__device__ __forceinline__ float softplusf(float x) { return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x)); }

template <int V, int kFlags>
__global__ void __launch_bounds__(kDecThreads, 2048 / kDecThreads / 4) kda_decode_kernel(const DecodeParams p) {
  // V / kDecRows CTAs per (sequence, head), V = 64, 128 or 256.  The CTA's kDecRows state
  // rows are block blockIdx.x of the [B * H * V / kDecRows, kDecRows, 128] state.
  constexpr int kSubs = V / kDecRows;
  const int sub = kSubs == 1 ? 0 : (int)(blockIdx.x % kSubs);
  const int nh = kSubs == 1 ? (int)blockIdx.x : (int)(blockIdx.x / kSubs);
  const int vbase = sub * kDecRows;   // value index of this CTA's first row
  const int n = nh / p.H, h = nh - n * p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ __align__(16) float s_alpha[128], s_kh[128], s_qh[128], s_v[kDecRows];
  __shared__ float s_norm[2][4];
  __shared__ float s_beta;

  // ---- the state rows of this warp, four key channels per lane (K = 64: lanes 16-31 hold
  //      the channels 64-127, which stay zero)
  constexpr int K = (kFlags & kDecK64) ? 64 : 128;       // key channels of the caller's tensors
  constexpr int kq = K / 4;                               // four-channel groups a state row holds
  const bool kl = lane < kq;                              // this lane's channels exist
  const size_t srow0 = (size_t)blockIdx.x * kDecRows;   // first state row of this CTA
  float4 st[kRowsPerWarp];
  if (p.state_dtype == 2) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.state) + srow0 * K);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
      st[r] = kl ? src[(kRowsPerWarp * warp + r) * kq + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    const uint2* src = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.state) + srow0 * K);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const uint2 w = kl ? src[(kRowsPerWarp * warp + r) * kq + lane] : make_uint2(0u, 0u);
      st[r] = make_float4(bf(w.x & 0xffffu), bf(w.x >> 16), bf(w.y & 0xffffu), bf(w.y >> 16));
    }
  }
  constexpr bool gate_pre = kFlags & kGatePreactivated;    // then A_log and dt_bias may be null
  const float rate = gate_pre ? 0.f : expf(p.A_log[h]);

#pragma unroll 1
  for (int t = 0; t < p.T; ++t) {
    const size_t tok = ((size_t)n * p.T + t) * p.H + h;   // row of [B*T, H]
    // ---- per-channel vectors of this token (threads 0-127, channel = tid)
    float kk = 0.f, qq = 0.f;
    if (tid < 128) {
      const bool ch = tid < K;   // channel tid exists (K = 64: channels 64-127 are zero)
      const float gt = ch ? bf(p.g[tok * K + tid]) : 0.f;
      float ghat = gt;
      if (!gate_pre && ch) {
        const float pre = gt + p.dt_bias[(size_t)h * K + tid];
        ghat = (kFlags & kGateSoftplus) ? -rate * softplusf(pre) : p.lower_bound * sigmoidf(rate * pre);
      }
      s_alpha[tid] = expf(ghat);
      kk = ch ? bf(p.k[tok * K + tid]) : 0.f;
      qq = ch ? bf(p.q[tok * K + tid]) : 0.f;
      s_kh[tid] = kk;
      s_qh[tid] = qq;
      if (tid < kDecRows) s_v[tid] = bf(p.v[tok * V + vbase + tid]);   // this CTA's rows' values
      const float sk = warp_sum(kk * kk), sq = warp_sum(qq * qq);
      if (lane == 0) {
        s_norm[0][warp] = sk;
        s_norm[1][warp] = sq;
      }
    }
    if (tid == 0) s_beta = (kFlags & kBetaPreactivated) ? bf(p.beta[tok]) : sigmoidf(bf(p.beta[tok]));
    __syncthreads();
    // ---- the rows: decay, delta update, output from the updated row (each lane
    //      normalises its own four channels of k and q)
    const float4 al = reinterpret_cast<const float4*>(s_alpha)[lane];
    float4 kh = reinterpret_cast<const float4*>(s_kh)[lane];
    float4 qh = reinterpret_cast<const float4*>(s_qh)[lane];
    if (!(kFlags & kNoQkL2Norm)) {
      const float rk = 1.f / sqrtf(s_norm[0][0] + s_norm[0][1] + s_norm[0][2] + s_norm[0][3] + 1e-6f);
      const float rq = 1.f / sqrtf(s_norm[1][0] + s_norm[1][1] + s_norm[1][2] + s_norm[1][3] + 1e-6f);
      kh.x *= rk; kh.y *= rk; kh.z *= rk; kh.w *= rk;
      qh.x *= rq; qh.y *= rq; qh.z *= rq; qh.w *= rq;
    }
    const float beta = s_beta;
    float d[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      st[r].x *= al.x; st[r].y *= al.y; st[r].z *= al.z; st[r].w *= al.w;
      d[r] = st[r].x * kh.x + st[r].y * kh.y + st[r].z * kh.z + st[r].w * kh.w;
    }
    warp_sum16(d);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const float c = beta * (s_v[kRowsPerWarp * warp + r] - d[r]);
      st[r].x = fmaf(c, kh.x, st[r].x); st[r].y = fmaf(c, kh.y, st[r].y);
      st[r].z = fmaf(c, kh.z, st[r].z); st[r].w = fmaf(c, kh.w, st[r].w);
      d[r] = st[r].x * qh.x + st[r].y * qh.y + st[r].z * qh.z + st[r].w * qh.w;
    }
    warp_sum16(d);
    if (lane < kRowsPerWarp) {
      float o = d[0];
#pragma unroll
      for (int r = 1; r < kRowsPerWarp; ++r) o = lane == r ? d[r] : o;
      p.out[tok * V + vbase + kRowsPerWarp * warp + lane] =
          __bfloat16_as_ushort(__float2bfloat16_rn(p.scale * o));
    }
    if (t + 1 < p.T) __syncthreads();   // the per-channel vectors are rewritten by the next token
  }

  // ---- write the rows back
  if (p.state_dtype == 2) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.state) + srow0 * K);
    if (kl) {
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) dst[(kRowsPerWarp * warp + r) * kq + lane] = st[r];
    }
  } else {
    uint2* dst = reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.state) + srow0 * K);
    if (kl) {
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
        dst[(kRowsPerWarp * warp + r) * kq + lane] =
            make_uint2(pack_bf16x2(st[r].x, st[r].y), pack_bf16x2(st[r].z, st[r].w));
    }
  }
}

}  // namespace

using DecodeKernel = void (*)(DecodeParams);

// One kernel per V and flag set, K = 64 as a flag bit (the preactivated and softplus gates
// exclude each other: no kernel for both)
template <int V, int F>
constexpr DecodeKernel decode_entry() {
  if constexpr ((F & kGatePreactivated) && (F & kGateSoftplus)) return nullptr;
  else return kda_decode_kernel<V, F>;
}
template <int V, int... F>
constexpr std::array<DecodeKernel, sizeof...(F)> decode_row(std::integer_sequence<int, F...>) {
  return {decode_entry<V, F>()...};
}
constexpr auto kDecodeV64 = decode_row<64>(std::make_integer_sequence<int, 2 * kDecK64>{});
constexpr auto kDecodeV128 = decode_row<128>(std::make_integer_sequence<int, 2 * kDecK64>{});
constexpr auto kDecodeV256 = decode_row<256>(std::make_integer_sequence<int, 2 * kDecK64>{});

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
  // p.vsplit carries V / 64 (1, 2 or 4): one 64-row CTA per 64 value rows
  const long long grid = (long long)p.B * p.H * p.vsplit;
  if (grid <= 0 || p.T <= 0) return cudaSuccess;
  // V, K and the flags are template parameters: the common case (K = V = 128, every step in
  // the kernel) carries no per-thread tests of any of them
  const int vi = p.vsplit == 1 ? 0 : (p.vsplit == 2 ? 1 : 2);
  const int f = (int)(p.flags & kValidFlags) | (p.kdim == 64 ? kDecK64 : 0);
  const DecodeKernel k = vi == 0 ? kDecodeV64[f] : (vi == 1 ? kDecodeV128[f] : kDecodeV256[f]);
  if (k == nullptr) return cudaErrorInvalidValue;
  k<<<(unsigned)grid, kDecThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
