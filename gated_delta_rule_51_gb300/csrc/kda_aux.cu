// kda_aux.cu -- device-side work scheduling and the segment-carry composition.
//
// Long sequences are cut into segments so that the sequential chunk recurrence of
// one (sequence, head) can run on several SMs at once.  Because a segment maps the
// state affinely, S_out = P S_in + Q, every segment first runs its forward pass from
// a known start (segment 0 from the true initial state, the others from zero), which
// writes its outputs and its local carry Q_s; segments 1 .. n-2 also run from the
// identity with zero values, which gives their transitions P_s.  The carries are then
// composed in order, S_{s+1} = P_s S_s + Q_s, and each segment s >= 1 finally runs a
// correction: the recurrence with zero values started from S_s, whose outputs are
// added to the ones already written (by linearity in (v, S_in) this is exactly the
// forward from the true state).  Transition and correction runs stop as soon as the
// state they carry is exactly zero in fp32 -- from then on it stays zero -- so for a
// gate that forgets, a split costs little more than the forward pass itself.  All of
// this is derived from the recurrence; FlashKDA's README carries the state across
// calls, with no segment scan.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

// ------------------------------------------------------------------ schedule
// One CTA.  Reads cu_seqlens (or the fixed batch layout), validates it, and
// writes the three work lists and their counts into the workspace.
//
// A sequence of len tokens is cut into nseg = ceil(len / L) segments of L tokens (the
// last one shorter).  Per head, the lists get:
//   transitions    T_s, s = 1 .. nseg-2: transition runs into slot P_s (with a zero flag);
//                  a launch of their own, first (they usually stop after a few chunks).
//   forward        F_s, s = 0 .. nseg-1: forward runs writing outputs; F_0 starts from
//                  the caller's initial state, the others from zero.  F_s stores its final
//                  state in slot Q_s (for s = nseg-1 only when there is a final state;
//                  an unsplit sequence writes the caller's final state directly).
//   compose        S_1 = Q_0; S_{s+1} = P_s S_s + Q_s into Q_s, s = 1 .. nseg-2.
//   last launch    C_s, s = 1 .. nseg-1: correction runs from Q_{s-1} = S_s, adding to the
//                  outputs of F_s; C_{nseg-1} writes the final state Q_{nseg-1} + D.
// Slots of one (sequence, head), from base = slot0 H + h 2 (nseg-1):
//   Q_s = base + s (s = 0 .. nseg-1),  P_s = base + nseg + s - 1 (s = 1 .. nseg-2).
constexpr int kSchedThreads = 1024;
static_assert(kSchedThreads == 32 * 32, "block_scan scans one total per warp in one warp");

__device__ __forceinline__ WorkItem make_item(long long row0, long long len, long long h, int mode, long long n,
                                              long long in_slot, long long out_slot, long long aux_slot) {
  WorkItem w;
  w.row0 = (int)row0;
  w.len = (int)len;
  w.head = (int)h;
  w.mode = mode;
  w.seq = (int)n;
  w.in_slot = (int)in_slot;
  w.out_slot = (int)out_slot;
  w.aux_slot = (int)aux_slot;
  return w;
}

// inclusive scan of one value per thread across the block: shuffles within each
// warp, then the 32 warp totals scanned by warp 0 (two block barriers in all)
__device__ long long block_scan(long long x, long long* buf) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long t = buf[lane];   // kSchedThreads / 32 == 32 warp totals
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    buf[lane] = t;
  }
  __syncthreads();
  const long long r = x + (warp > 0 ? buf[warp - 1] : 0);
  __syncthreads();   // buf is reused by the next scan
  return r;
}

// The forward runs are listed longest first, so that the first wave puts the longest runs one
// to an SM and the short ones fill the second CTA slots and finish early: the long chains then
// run alone for most of their length.  Runs are ranked by a length bucket, four buckets per
// octave of chunk count (ties in arbitrary order; every run computes the same either way).
constexpr int kLenBuckets = 4 * 32;
constexpr int kSegCandidates = 64;   // segment lengths the schedule weighs against one wave
__device__ __forceinline__ int len_bucket(long long chunks) {
  if (chunks < 4) return (int)(chunks < 0 ? 0 : chunks);
  const int msb = 63 - __clzll(chunks);
  return 4 * msb + (int)((chunks >> (msb - 2)) & 3);
}

__global__ void __launch_bounds__(kSchedThreads) kda_schedule_kernel(const ScheduleParams p) {
  __shared__ unsigned int s_hist[kLenBuckets];
  __shared__ long long s_buf[kSchedThreads];
  __shared__ long long s_tot[6];   // runs, corrections, compose chains, slots, transitions, forward runs
  __shared__ int s_start[kSchedThreads], s_len[kSchedThreads], s_nseg[kSchedThreads], s_incl[kSchedThreads];
  __shared__ long long s_run0[kSchedThreads], s_corr0[kSchedThreads], s_slot0[kSchedThreads], s_tr0[kSchedThreads];
  __shared__ int s_comp0[kSchedThreads];
  __shared__ int s_err;
  __shared__ unsigned long long s_max_chunks, s_sum_chunks;
  __shared__ unsigned long long s_runs[kSegCandidates];
  __shared__ long long s_L;
  const int tid = threadIdx.x;
  const long long H = p.H;
  const long long total_rows = p.B * p.T;
  if (tid == 0) {
    s_err = 0;
    s_max_chunks = 0;
    s_sum_chunks = 0;
  }
  for (int i = tid; i < kLenBuckets; i += kSchedThreads) s_hist[i] = 0;
  for (int i = tid; i < kMaxSmIds; i += kSchedThreads) p.sm_arrivals[i] = 0;
  if (tid < 3) p.hdr->take[tid] = 0;
  __syncthreads();
  // Split long sequences when the longest would outlast the mean load of a resident CTA by
  // more than a quarter.  A split costs, per extra segment, a transition run and a correction
  // run; both stop as soon as what they carry is exactly zero in fp32, which for a gate that
  // forgets comes after a few chunks (a gate that keeps everything makes them full passes).
  if (!p.seg_forced && p.seg_tokens < total_rows) {
    unsigned long long mx = 0, sum = 0;
    for (long long n = tid; n < p.N; n += kSchedThreads) {
      long long len = p.T;
      if (p.cu_seqlens) {
        long long a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
        a = a < 0 ? 0 : (a > total_rows ? total_rows : a);
        b = b < a ? a : (b > total_rows ? total_rows : b);
        len = b - a;
      }
      const unsigned long long c = (unsigned long long)((len + 15) / 16);
      mx = c > mx ? c : mx;
      sum += c;
    }
    atomicMax(&s_max_chunks, mx);
    atomicAdd(&s_sum_chunks, sum);
  }
  __syncthreads();
  if (tid == 0) {
    long long Lx = p.seg_tokens;
    if (!p.seg_forced && p.seg_tokens < total_rows) {
      const long long per_cta = ((long long)s_sum_chunks * H + p.resident - 1) / p.resident;
      if (4 * (long long)s_max_chunks <= 5 * per_cta) Lx = (total_rows + 15) / 16 * 16;   // no split
    }
    s_L = Lx;
  }
  __syncthreads();
  // A split whose forward runs only just exceed one wave of resident CTAs (by at most a quarter)
  // leaves the excess runs for a second wave, each after a whole run of the first: take instead
  // the shortest longer segment, at most a quarter longer, whose runs fit one wave.  Candidates
  // L0 + c * step (kSegCandidates of them) are counted side by side.  Longer segments only mean
  // fewer runs, so the work lists sized from the host's length still suffice.
  if (!p.seg_forced && s_L < total_rows) {
    const long long L0 = s_L;
    long long step = ((L0 / 4) / kSegCandidates + 15) / 16 * 16;
    if (step < 16) step = 16;
    for (int i = tid; i < kSegCandidates; i += kSchedThreads) s_runs[i] = 0;
    __syncthreads();
    for (long long idx = tid; idx < (long long)p.N * kSegCandidates; idx += kSchedThreads) {
      const long long n = idx / kSegCandidates;
      const int c = (int)(idx - n * kSegCandidates);
      long long len = p.T;
      if (p.cu_seqlens) {
        long long a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
        a = a < 0 ? 0 : (a > total_rows ? total_rows : a);
        b = b < a ? a : (b > total_rows ? total_rows : b);
        len = b - a;
      }
      const long long Lc = L0 + c * step;
      atomicAdd(&s_runs[c], (unsigned long long)(len <= 0 ? 1 : (len + Lc - 1) / Lc));
    }
    __syncthreads();
    if (tid == 0) {
      const long long runs0 = (long long)s_runs[0] * H;
      if (runs0 > p.resident && 4 * runs0 <= 5 * p.resident) {
        for (int c = 1; c < kSegCandidates; ++c) {
          const long long Lc = L0 + c * step;
          if (4 * Lc > 5 * L0) break;
          if ((long long)s_runs[c] * H <= p.resident) {
            s_L = Lc;
            break;
          }
        }
      }
    }
    __syncthreads();
  }
  const long long L = s_L;
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1 && tid == 0) {   // bucket counts -> first rank of each bucket, longest first
      unsigned int start = 0;
      for (int bk = kLenBuckets - 1; bk >= 0; --bk) {
        const unsigned int c = s_hist[bk];
        s_hist[bk] = start;
        start += c;
      }
    }
    if (tid == 0) s_tot[0] = s_tot[1] = s_tot[2] = s_tot[3] = s_tot[4] = s_tot[5] = 0;
    __syncthreads();
    for (long long base = 0; base < p.N; base += kSchedThreads) {
      const long long n = base + tid;
      long long start = 0, len = 0, nseg = 0;
      if (n < p.N) {
        if (p.cu_seqlens) {
          long long a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
          if ((n == 0 && a != 0) || b < a || (n == p.N - 1 && b != total_rows)) s_err = 1;
          a = a < 0 ? 0 : (a > total_rows ? total_rows : a);
          b = b < a ? a : (b > total_rows ? total_rows : b);
          start = a;
          len = b - a;
        } else {
          start = n * p.T;
          len = p.T;
        }
        nseg = len <= 0 ? 1 : (len + L - 1) / L;
      }
      const long long ntr = nseg >= 3 ? nseg - 2 : 0;
      const long long nruns = nseg + ntr;
      const long long ncorr = nseg >= 2 ? nseg - 1 : 0;
      const long long ncomp = nseg >= 3 ? 1 : 0;
      const long long nslot = nseg >= 2 ? 2 * (nseg - 1) : 0;
      const long long incl = block_scan(nruns, s_buf);
      const long long run0 = s_tot[0] + incl - nruns;
      // pass 0: histogram of the forward runs' lengths; pass 1: each forward run's rank
      if (n < p.N) {
        for (long long r = 0; r < nseg; ++r) {
          const long long flen = len <= 0 ? 0 : (len - r * L < L ? len - r * L : L);
          const int bk = len_bucket((flen + 15) / 16);
          if (pass == 0) atomicAdd(&s_hist[bk], 1u);
          else if (run0 + r < p.cap_ranks) p.seg_rank[run0 + r] = (int)atomicAdd(&s_hist[bk], 1u);
        }
      }
      const long long tr0 = s_tot[4] + block_scan(ntr, s_buf) - ntr;
      const long long fw0 = s_tot[5] + block_scan(nseg, s_buf) - nseg;
      const long long corr0 = s_tot[1] + block_scan(ncorr, s_buf) - ncorr;
      const long long comp0 = s_tot[2] + block_scan(ncomp, s_buf) - ncomp;
      const long long slot0 = s_tot[3] + block_scan(nslot, s_buf) - nslot;
      const int count = (int)(p.N - base < kSchedThreads ? p.N - base : kSchedThreads);
      if (pass == 1) {
        s_start[tid] = (int)start;
        s_len[tid] = (int)len;
        s_nseg[tid] = (int)nseg;
        s_incl[tid] = (int)incl;
        s_run0[tid] = run0;
        s_corr0[tid] = corr0;
        s_comp0[tid] = (int)comp0;
        s_slot0[tid] = slot0;
        s_tr0[tid] = tr0;
        __syncthreads();
        // every (head, run) of this tile's sequences, spread over all threads
        const long long tile_runs = s_incl[count - 1];
        const long long in_user = p.has_init ? kInUser : kInZero;
        for (long long idx = tid; idx < tile_runs * H; idx += kSchedThreads) {
          const long long h = idx / tile_runs;
          const int rl = (int)(idx - h * tile_runs);
          int lo = 0, hi = count - 1;                 // first sequence with s_incl > rl
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_incl[mid] > rl) hi = mid; else lo = mid + 1;
          }
          const int nl = lo;
          const long long ns = s_nseg[nl];
          const long long nr = ns + (ns >= 3 ? ns - 2 : 0);
          const long long r = rl - (s_incl[nl] - nr);
          const long long st0 = s_start[nl], ln = s_len[nl];
          const long long nn = base + nl;
          const long long gr = s_run0[nl] + r;
          const long long fi = (gr < p.cap_ranks ? (long long)p.seg_rank[gr] : gr) * H + h;
          const long long qb = s_slot0[nl] * H + h * 2 * (ns - 1);   // Q_0 (split sequences)
          const bool slots_ok = ns < 2 || qb + 2 * (ns - 1) <= p.cap_slots;
          if (r < ns) {
            const long long s = r;
            const long long flen = ln <= 0 ? 0 : (ln - s * L < L ? ln - s * L : L);
            long long out_slot;
            if (ns == 1) out_slot = p.has_final ? kOutUser : kOutNone;
            else out_slot = (s <= ns - 2 || p.has_final) ? qb + s : kOutNone;
            if (fi < p.cap_forward && slots_ok)
              p.forward[fi] = make_item(st0 + s * L, flen, h, kModeForward, nn, s == 0 ? in_user : kInZero, out_slot,
                                        -1);
            if (s >= 1) {
              const long long ci = (s_corr0[nl] + s - 1) * H + h;
              const bool fin = s == ns - 1 && p.has_final;
              if (ci < p.cap_correct && slots_ok)
                p.correct[ci] = make_item(st0 + s * L, flen, h, kModeCorrect, nn, qb + s - 1,
                                          fin ? kOutUser : kOutNone, fin ? qb + s : -1);
            }
            if (s == 0 && ns >= 3) {
              const long long ci = (long long)s_comp0[nl] * H + h;
              if (ci < p.cap_compose && slots_ok) {
                ComposeItem it;
                it.head = (int)h;
                it.first_q_slot = (int)qb;
                it.first_p_slot = (int)(qb + ns);
                it.n_steps = (int)(ns - 2);
                p.compose[ci] = it;
              }
            }
          } else {
            const long long s = r - ns + 1;   // transition of segment s, 1 <= s <= ns - 2
            const long long ti = (s_tr0[nl] + s - 1) * H + h;
            if (ti < p.cap_transition && slots_ok)
              p.transition[ti] = make_item(st0 + s * L, L, h, kModeTransition, nn, kInIdentity, qb + ns + s - 1, -1);
          }
        }
      }
      __syncthreads();
      if (tid == kSchedThreads - 1) {
        s_tot[0] = run0 + nruns;
        s_tot[1] = corr0 + ncorr;
        s_tot[2] = comp0 + ncomp;
        s_tot[3] = slot0 + nslot;
        s_tot[4] = tr0 + ntr;
        s_tot[5] = fw0 + nseg;
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    const long long nf = s_tot[5] * H;
    const long long nt = s_tot[4] * H;
    const long long nc = s_tot[1] * H;
    const long long ncm = s_tot[2] * H;
    p.hdr->n_forward = (int)(nf < p.cap_forward ? nf : p.cap_forward);
    p.hdr->n_transition = (int)(nt < p.cap_transition ? nt : p.cap_transition);
    p.hdr->n_correct = (int)(nc < p.cap_correct ? nc : p.cap_correct);
    p.hdr->n_compose = (int)(ncm < p.cap_compose ? ncm : p.cap_compose);
    p.hdr->err = s_err ? kErrBadSeqlens : 0;
  }
}

cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t s) {
  kda_schedule_kernel<<<1, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ compose
// S^T_{s+1} = S^T_s P^T_s + Q^T_s, all 128 x 128 fp32 in the [V, K] layout:
// out[v][k] = sum_m in[v][m] * Pst[m][k] + Qst[v][k] where Pst is the stored
// transition slot (row m = column m of P).  Rows of S^T are independent, so
// each CTA owns kRows (16 or 32) rows of one (sequence, head) chain and walks its segments:
// S_{s+1} = S_s P_s + Q_s on its rows.  The chain is sequential, so each step's
// operands (the 64 KiB transition P_s and the CTA's 8 KiB of Q_s) are brought into
// shared memory by bulk copies one step ahead, while the current step computes.
// Each thread computes kRows / 4 rows x 2 columns: per m, float4s of S (kept
// transposed, St[m][v]) and one float2 of P feed the FMAs.  32-row CTAs are used when
// 16-row ones would not all fit on the GPU at once (one CTA per SM: the double-buffered
// transition takes 128 KiB).
constexpr int kComposeThreads = 256;
constexpr uint32_t kPBytes = 128 * 128 * 4;

template <int kRows>
struct ComposeSmem {
  static constexpr int kPitch = kRows + 4;   // floats per St row (16-byte aligned, spreads banks)
  float P[2][128][128];
  float Q[2][kRows][128];
  float St[128][kPitch];   // this CTA's rows of S^T, transposed: St[m][v]
};

__device__ __forceinline__ void bulk_load_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int kRows>
__global__ void __launch_bounds__(kComposeThreads) kda_compose_kernel(const ComposeParams p) {
  // the correction launch after this one may start beside it: its runs read the composed
  // states only after waiting for this grid
  griddep_launch_dependents();
  constexpr int kRowsPerThread = kRows / 4;
  constexpr uint32_t kQBytes = kRows * 128 * 4;
  const int item = blockIdx.x / (128 / kRows);
  const int part = blockIdx.x % (128 / kRows);
  if (item >= *p.item_count) return;
  const ComposeItem ci = p.items[item];
  extern __shared__ __align__(128) uint8_t csm[];
  ComposeSmem<kRows>& S = *reinterpret_cast<ComposeSmem<kRows>*>(csm);
  __shared__ __align__(8) uint64_t bar[2];
  const int tid = threadIdx.x;
  const int k2 = 2 * (tid & 63);                // columns k2, k2 + 1
  const int r4 = kRowsPerThread * (tid >> 6);   // rows r4 .. r4 + kRowsPerThread - 1 of this CTA's
  const int v0 = part * kRows;
  float* slots = p.ws_states;
  auto P_src = [&](int st) { return slots + (size_t)(ci.first_p_slot + st - 1) * 16384; };
  auto Q_row0 = [&](int st) { return slots + (size_t)(ci.first_q_slot + st) * 16384 + (size_t)v0 * 128; };
  // a transition its run found exactly zero: S_{s+1} = Q_s, already in place
  auto zero_p = [&](int st) { return p.zero_flags[ci.first_p_slot + st - 1] != 0; };
  auto fetch = [&](int st) {   // operands of step st into buffer st & 1 (thread 0)
    uint64_t* b = &bar[st & 1];
    const bool z = zero_p(st);
    mbar_arrive_expect_tx(b, (z ? 0u : kPBytes) + kQBytes);
    if (!z) bulk_load_g2s(&S.P[st & 1][0][0], P_src(st), kPBytes, b);
    bulk_load_g2s(&S.Q[st & 1][0][0], Q_row0(st), kQBytes, b);
  };
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  // S_1 = Q slot 0 (already the true state after segment 0)
  for (int i = tid; i < kRows * 128; i += kComposeThreads)
    S.St[i % 128][i / 128] = slots[(size_t)ci.first_q_slot * 16384 + (size_t)(v0 + i / 128) * 128 + i % 128];
  __syncthreads();
  if (tid == 0) {
    if (ci.n_steps >= 1) fetch(1);
    if (ci.n_steps >= 2) fetch(2);
  }
  for (int st = 1; st <= ci.n_steps; ++st) {
    const int b = st & 1;
    {
      const long long t0 = clock64();   // bounded: the copy always lands; the data is garbage otherwise
      while (!mbar_try_wait(&bar[b], ((st - 1) >> 1) & 1))
        if (clock64() - t0 > kWaitTimeoutCycles) break;
    }
    float2 acc[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) acc[i] = *reinterpret_cast<const float2*>(&S.Q[b][r4 + i][k2]);
    const bool z = zero_p(st);
    if (!z) {
#pragma unroll 8
      for (int m = 0; m < 128; ++m) {
        const float2 pm = *reinterpret_cast<const float2*>(&S.P[b][m][k2]);
#pragma unroll
        for (int i4 = 0; i4 < kRowsPerThread; i4 += 4) {
          const float4 sv = *reinterpret_cast<const float4*>(&S.St[m][r4 + i4]);
          const float s4[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[i4 + i].x = fmaf(s4[i], pm.x, acc[i4 + i].x);
            acc[i4 + i].y = fmaf(s4[i], pm.y, acc[i4 + i].y);
          }
        }
      }
    }
    __syncthreads();   // every thread is done with St and with buffer b
    float* Q = Q_row0(st);
#pragma unroll
    for (int i4 = 0; i4 < kRowsPerThread; i4 += 4) {
      *reinterpret_cast<float4*>(&S.St[k2][r4 + i4]) =
          make_float4(acc[i4].x, acc[i4 + 1].x, acc[i4 + 2].x, acc[i4 + 3].x);
      *reinterpret_cast<float4*>(&S.St[k2 + 1][r4 + i4]) =
          make_float4(acc[i4].y, acc[i4 + 1].y, acc[i4 + 2].y, acc[i4 + 3].y);
    }
    if (!z) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) *reinterpret_cast<float2*>(&Q[(size_t)(r4 + i) * 128 + k2]) = acc[i];
    }
    if (tid == 0 && st + 2 <= ci.n_steps) {
      fence_proxy_async_smem();   // the generic reads of buffer b are ordered before the refill
      fetch(st + 2);
    }
    __syncthreads();
  }
}

size_t compose_smem_bytes() { return sizeof(ComposeSmem<32>); }

// grid: compose items (chains); sms: SMs of the device
cudaError_t launch_compose(const ComposeParams& p, int grid, int sms, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  // 16-row CTAs while they fit on the GPU at once, else 32-row ones (half the CTAs)
  const bool wide = (long long)grid * (128 / 16) > (long long)sms;
  const int smem = wide ? (int)sizeof(ComposeSmem<32>) : (int)sizeof(ComposeSmem<16>);
  const auto kernel = wide ? kda_compose_kernel<32> : kda_compose_kernel<16>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid * (128 / (wide ? 32 : 16)), kComposeThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
