// kda_api.cu -- the C ABI (include/kda.h): argument checks, workspace layout,
// TMA descriptors and the launch sequence of the KDA forward pass.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"

using namespace kda;

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kSlotBytes = 128 * 128 * sizeof(float);

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

// Attributes of the current device, queried once per device and cached (every call
// needs them; the queries cost more than the rest of the host-side work).
kda_status device_info(DeviceInfo* out) {
  constexpr int kMaxDevices = 64;
  static DeviceInfo cache[kMaxDevices];
  static std::atomic<bool> have[kMaxDevices];
  static std::mutex fill;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable && have[dev].load(std::memory_order_acquire)) {
    *out = cache[dev];
    return KDA_OK;
  }
  DeviceInfo d;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (cacheable) {
    std::lock_guard<std::mutex> lock(fill);
    cache[dev] = d;
    have[dev].store(true, std::memory_order_release);
  }
  *out = d;
  return KDA_OK;
}

// Segment length set through the environment (tests and tuning), else 0.
int64_t forced_seg_tokens() {
  const char* env = std::getenv("KDA_SEG_TOKENS");
  if (env == nullptr) return 0;
  const long long v = std::atoll(env);
  return v >= 16 ? (v + 15) / 16 * 16 : 0;
}

// Tokens per segment.  A (sequence, head) chain is sequential over its chunks;
// when there are too few chains to fill the GPU, long sequences are cut into
// segments so that about one wave of forward work items exists.  Segments are
// at least 512 tokens; the value is a multiple of 16.  This is an upper bound on
// the length the schedule kernel uses (it never cuts shorter, so the work-list
// capacities sized from it always suffice).
int64_t choose_seg_tokens(const kda_shape& s, int sms) {
  const int64_t rows = s.B * s.T;
  if (const int64_t f = forced_seg_tokens()) return f;
  const int64_t resident = 2 * (int64_t)std::max(sms, 1);   // CTAs resident at once
  const int64_t chains = s.N * s.H;
  const int64_t no_split = std::max<int64_t>(16, (rows + 15) / 16 * 16);
  if (chains >= 2 * resident || rows == 0) return no_split;
  int64_t L = (rows * s.H + resident - 1) / resident;
  L = std::max<int64_t>(512, (L + 15) / 16 * 16);
  return std::min(L, no_split);
}

struct Layout {
  int64_t seg_tokens = 0;
  int64_t cap_forward = 0, cap_transition = 0, cap_correct = 0, cap_compose = 0, cap_slots = 0, cap_ranks = 0;
  size_t off_hdr = 0, off_forward = 0, off_transition = 0, off_correct = 0, off_compose = 0, off_slots = 0,
         off_ranks = 0, off_sm = 0, off_zero = 0;
  size_t total = 0;
};

Layout make_layout(const kda_shape& s, int sms) {
  Layout L;
  const int64_t rows = s.B * s.T;
  L.seg_tokens = choose_seg_tokens(s, sms);
  const int64_t splits = rows / L.seg_tokens;   // bound on sum over sequences of (nseg - 1)
  // nseg forward and (nseg - 2) transition runs per sequence (the ranks are indexed over both)
  L.cap_ranks = s.N + 2 * splits;
  L.cap_forward = s.H * (s.N + splits);
  L.cap_transition = s.H * splits;
  L.cap_correct = s.H * splits;                 // nseg - 1 per sequence
  L.cap_slots = 2 * s.H * splits;               // 2 (nseg - 1) per split sequence
  L.cap_compose = s.H * std::min<int64_t>(s.N, splits);
  size_t off = 0;
  L.off_hdr = off;
  off = align_up(off + sizeof(WorkHeader));
  L.off_forward = off;
  off = align_up(off + (size_t)L.cap_forward * sizeof(WorkItem));
  L.off_transition = off;
  off = align_up(off + (size_t)L.cap_transition * sizeof(WorkItem));
  L.off_correct = off;
  off = align_up(off + (size_t)L.cap_correct * sizeof(WorkItem));
  L.off_compose = off;
  off = align_up(off + (size_t)L.cap_compose * sizeof(ComposeItem));
  L.off_ranks = off;
  off = align_up(off + (size_t)L.cap_ranks * sizeof(int));
  L.off_sm = off;
  off = align_up(off + (size_t)kMaxSmIds * sizeof(int));
  L.off_zero = off;
  off = align_up(off + (size_t)L.cap_slots * sizeof(int));
  L.off_slots = off;
  off = align_up(off + (size_t)L.cap_slots * kSlotBytes);
  L.total = off;
  return L;
}

// The backward pass's workspace: header (error word), per token-head prepared vectors,
// the stored states, the row-slice partials, the per-token dA_log terms and the
// parameter-reduction blocks.
struct BwdLayout {
  size_t off_hdr = 0, off_prep = 0, off_ckpt = 0, off_part = 0, off_dA = 0, off_ppart = 0, total = 0;
  int nblk = 0;
};

BwdLayout make_bwd_layout(const kda_shape& s) {
  BwdLayout L;
  const size_t BT = (size_t)(s.B * s.T), TH = BT * (size_t)s.H;
  const size_t nslot = BT / kBwdChunk + (size_t)s.N + 1;
  L.nblk = (int)((BT + kBwdParamTokens - 1) / kBwdParamTokens);
  size_t off = 0;
  L.off_hdr = off;
  off = align_up(off + sizeof(WorkHeader));
  L.off_prep = off;
  off = align_up(off + TH * kBwdRowStride * sizeof(float));
  L.off_ckpt = off;
  off = align_up(off + nslot * (size_t)s.H * kSlotBytes);
  L.off_part = off;
  off = align_up(off + (size_t)kBwdSlices * TH * kBwdRowStride * sizeof(float));
  L.off_dA = off;
  off = align_up(off + TH * sizeof(float));
  L.off_ppart = off;
  off = align_up(off + (size_t)L.nblk * (size_t)s.H * kBwdParamStride * sizeof(float));
  L.total = off;
  return L;
}

// The chunked backward's workspace: header, the chains' runs and correction runs, the state
// slots of cut sequences (2 kBwdMaxParts - 1 per (sequence, head), for at most
// kBwdMaxSplitChains chains: more chains are never cut), per (chunk slot, head) the stored states (bf16),
// Vn and dVn (fp32), the state products and the parameter partials, then the partials of blocks of
// 64 slots.  Slots: n + row0(n) / 16 + c is below N + B T / 16 + 1.
struct BwdChunkedLayout {
  size_t off_hdr = 0, off_items = 0, off_citems = 0, off_bslots = 0, off_s0 = 0, off_ds1 = 0, off_vn = 0, off_dvn = 0,
         off_xp = 0, off_zs = 0, off_ppart = 0, total = 0;
  int64_t nslots = 0;
  int nblk = 0;
};

BwdChunkedLayout make_bwd_chunked_layout(const kda_shape& s) {
  BwdChunkedLayout L;
  const size_t BT = (size_t)(s.B * s.T);
  L.nslots = (int64_t)(BT / 16) + s.N + 1;
  const size_t SH = (size_t)L.nslots * (size_t)s.H;
  L.nblk = (int)((BT + kBwdParamTokens - 1) / kBwdParamTokens);
  size_t off = 0;
  L.off_hdr = off;
  off = align_up(off + sizeof(WorkHeader));
  L.off_items = off;
  const size_t NH = (size_t)s.N * (size_t)s.H;
  off = align_up(off + 2 * kBwdMaxParts * NH * sizeof(WorkItem));
  L.off_citems = off;
  off = align_up(off + 2 * (kBwdMaxParts - 1) * NH * sizeof(WorkItem));
  L.off_bslots = off;
  off = align_up(off + (2 * kBwdMaxParts - 1) * std::min<size_t>(NH, kBwdMaxSplitChains) * kSlotBytes);
  L.off_s0 = off;
  off = align_up(off + SH * 16384 * sizeof(uint16_t));
  L.off_ds1 = off;
  off = align_up(off + SH * 16384 * sizeof(uint16_t));
  L.off_vn = off;
  off = align_up(off + SH * 2048 * sizeof(float));
  L.off_dvn = off;
  off = align_up(off + SH * 2048 * sizeof(float));
  L.off_xp = off;
  off = align_up(off + SH * 6144 * sizeof(float));
  L.off_zs = off;
  off = align_up(off + SH * 128 * sizeof(float));
  L.off_ppart = off;   // per (chunk slot, head) parameter partials, then per block of 64 slots
  off = align_up(off + ((size_t)std::max<int64_t>(L.nslots, 1) + (size_t)(L.nslots + 63) / 64) * (size_t)s.H *
                           kBwdParamStride * sizeof(float));
  L.total = off;
  return L;
}

kda_status check_shape(const kda_shape* s) {
  if (s == nullptr) return KDA_ERR_INVALID_ARGUMENT;
  if ((s->K != 64 && s->K != 128) || (s->V != 64 && s->V != 128 && s->V != 256)) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (s->B < 0 || s->T < 0 || s->H <= 0 || s->N < 0) return KDA_ERR_INVALID_ARGUMENT;
  if (s->B > 0 && s->T > (int64_t)0x7fffffff / std::max<int64_t>(s->B, 1)) return KDA_ERR_INVALID_ARGUMENT;
  const int64_t Hv = s->H * std::max<int64_t>(s->V / 128, 1);
  if (Hv > 65535 || s->N > (int64_t)0x7fffffff / Hv) return KDA_ERR_INVALID_ARGUMENT;
  return KDA_OK;
}

// The value columns of a state are independent, so V = 256 runs as two chains of
// 128 state rows per head: the work lists, segment slots and split policy see
// H x V/128 "heads" of width 128.  V = 64 runs as one chain whose rows 64-127 stay zero,
// and K = 64 as a chain whose channels 64-127 are zero.
kda_shape chain_shape(const kda_shape& s) {
  kda_shape c = s;
  c.H = s.H * std::max<int64_t>(s.V / 128, 1);
  c.K = 128;
  c.V = 128;
  return c;
}

cudaEvent_t g_profile_events[4] = {nullptr, nullptr, nullptr, nullptr};
bool g_profile = false;
thread_local int t_last_launches = 0;

// Inside a stream capture the record is external, so that a call captured into a CUDA
// graph records the event each time the graph runs; outside it is a plain record.  A
// profiling mark never fails the call: an error of its own is cleared at once.
void mark(int i, cudaStream_t s) {
  if (!g_profile || g_profile_events[i] == nullptr) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e == cudaSuccess)
    e = cs == cudaStreamCaptureStatusActive
            ? cudaEventRecordWithFlags(g_profile_events[i], s, cudaEventRecordExternal)
            : cudaEventRecord(g_profile_events[i], s);
  if (e != cudaSuccess) (void)cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [rows, H, width] bf16 viewed as a 3-D tensor {width, H, rows}; box {64, 1, 16}, 128-byte
// swizzle (width 128 for q and k, 64 for a V = 64 v).
bool encode_tile_map(CUtensorMap* m, const void* base, int64_t rows, int64_t H, int64_t width = 128) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)std::max<int64_t>(rows, 1)};
  cuuint64_t strides[2] = {(cuuint64_t)(width * 2), (cuuint64_t)(H * width * 2)};
  cuuint32_t box[3] = {64, 1, 16};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tensor seen as 4-D {64, H, rows, width / 64}: the 64-channel pieces of a row
// become the outermost dimension, so box {64, 1, 16, 2} lands in shared memory as
// [piece][16 rows][64 channels] -- two consecutive swizzled tiles -- in one copy.
// `width` is the row length in elements (128, or V for v): its 64-channel pieces are
// the outermost dimension, and a box takes two consecutive pieces.
bool encode_halves_map(CUtensorMap* m, const void* base, int64_t rows, int64_t H, int64_t width = 128) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)H, (cuuint64_t)std::max<int64_t>(rows, 1), (cuuint64_t)(width / 64)};
  cuuint64_t strides[3] = {(cuuint64_t)(width * 2), (cuuint64_t)(H * width * 2), 128};
  cuuint32_t box[4] = {64, 1, 16, 2};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KDA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K must be 64 or 128, V 64, 128 or 256)";
    case KDA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KDA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "a device-side wait timed out";
    case KDA_ERR_BAD_SEQLENS: return "malformed cu_seqlens";
    case KDA_ERR_GATE_RANGE: return "a chunk's decay left the chunked form's range (reserved; no longer raised)";
  }
  return "unknown status";
}

kda_status kda_workspace_size(const kda_shape* shape, size_t* bytes) {
  if (bytes == nullptr) return KDA_ERR_INVALID_ARGUMENT;
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  DeviceInfo d;
  if (device_info(&d) != KDA_OK) d.sms = 152;   // sizing only; kda_fwd checks the device
  *bytes = make_layout(chain_shape(*shape), d.sms).total;
  return KDA_OK;
}

// kda_flags: known bits only, and the preactivated and softplus gates exclude each other
static bool valid_flags(unsigned flags) {
  if (flags & ~(kda::kValidFlags | (unsigned)KDA_PRECISE_STATE)) return false;
  return !((flags & KDA_GATE_PREACTIVATED) && (flags & KDA_GATE_SOFTPLUS));
}
// only the in-kernel safe gate reads lower_bound
static bool uses_lower_bound(unsigned flags) { return !(flags & (KDA_GATE_PREACTIVATED | KDA_GATE_SOFTPLUS)); }

kda_status kda_decode(const kda_shape* shape, const void* q, const void* k, const void* v, const void* g,
                      const void* beta, float scale, void* out, const float* A_log, const float* dt_bias,
                      float lower_bound, void* state, kda_state_dtype state_dtype, unsigned flags,
                      kda_stream_t stream_) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  const kda_shape s = *shape;
  if (s.N != s.B) return KDA_ERR_INVALID_ARGUMENT;
  if ((long long)s.B * s.H * (s.V / 64) > 0x7fffffffLL) return KDA_ERR_INVALID_ARGUMENT;
  if (!valid_flags(flags)) return KDA_ERR_INVALID_ARGUMENT;
  const bool gate_here = !(flags & KDA_GATE_PREACTIVATED);
  if (uses_lower_bound(flags) && !(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_INVALID_ARGUMENT;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (s.B * s.T > 0) {
    const void* tok[] = {q, k, v, g, beta, out};
    for (const void* p : tok)
      if (p == nullptr || !aligned(p, 2)) return KDA_ERR_INVALID_ARGUMENT;
  }
  if (gate_here && (A_log == nullptr || dt_bias == nullptr || !aligned(A_log, 4) || !aligned(dt_bias, 4)))
    return KDA_ERR_INVALID_ARGUMENT;
  if (state_dtype != KDA_STATE_BF16 && state_dtype != KDA_STATE_FP32) return KDA_ERR_INVALID_ARGUMENT;
  if (s.B > 0 && (state == nullptr || !aligned16(state))) return KDA_ERR_INVALID_ARGUMENT;
  DeviceInfo d;
  if (device_info(&d) != KDA_OK) return KDA_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return KDA_ERR_UNSUPPORTED_DEVICE;
  DecodeParams dp;
  dp.q = static_cast<const uint16_t*>(q);
  dp.k = static_cast<const uint16_t*>(k);
  dp.v = static_cast<const uint16_t*>(v);
  dp.g = static_cast<const uint16_t*>(g);
  dp.beta = static_cast<const uint16_t*>(beta);
  dp.out = static_cast<uint16_t*>(out);
  dp.A_log = A_log;
  dp.dt_bias = dt_bias;
  dp.state = state;
  dp.state_dtype = state_dtype == KDA_STATE_FP32 ? 2 : 1;
  dp.B = (int)s.B;
  dp.T = (int)s.T;
  dp.H = (int)s.H;
  dp.vsplit = (int)(s.V / 64);   // 64-row CTAs per head
  dp.kdim = (int)s.K;
  dp.scale = scale;
  dp.lower_bound = lower_bound;
  dp.flags = (int)(flags & kValidFlags);
  if (launch_decode(dp, reinterpret_cast<cudaStream_t>(stream_)) != cudaSuccess) return KDA_ERR_CUDA;
  return KDA_OK;
}

kda_status kda_fwd(const kda_shape* shape, const void* q, const void* k, const void* v, const void* g,
                   const void* beta, float scale, void* out, const float* A_log, const float* dt_bias,
                   float lower_bound, const void* initial_state, kda_state_dtype init_dtype, void* final_state,
                   kda_state_dtype final_dtype, const int64_t* cu_seqlens, void* workspace,
                   size_t workspace_bytes, kda_stream_t stream) {
  return kda_fwd_ex(shape, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, init_dtype,
                    final_state, final_dtype, cu_seqlens, 0u, workspace, workspace_bytes, stream);
}

kda_status kda_fwd_ex(const kda_shape* shape, const void* q, const void* k, const void* v, const void* g,
                      const void* beta, float scale, void* out, const float* A_log, const float* dt_bias,
                      float lower_bound, const void* initial_state, kda_state_dtype init_dtype, void* final_state,
                      kda_state_dtype final_dtype, const int64_t* cu_seqlens, unsigned flags, void* workspace,
                      size_t workspace_bytes, kda_stream_t stream_) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  const kda_shape s = *shape;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // FlashKDA README, "Kernel API": a varlen call (cu_seqlens given) takes a batch of one row;
  // otherwise every one of the B rows is its own sequence (N = B).
  if (cu_seqlens != nullptr) {
    if (s.B != 1 || s.N < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (s.N == 0 && s.T != 0) return KDA_ERR_INVALID_ARGUMENT;
  } else if (s.N != s.B) {
    return KDA_ERR_INVALID_ARGUMENT;
  }
  if (!valid_flags(flags)) return KDA_ERR_INVALID_ARGUMENT;
  const bool gate_here = !(flags & KDA_GATE_PREACTIVATED);
  if (uses_lower_bound(flags) && !(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_INVALID_ARGUMENT;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
  const int64_t rows = s.B * s.T;
  // q, k, g, v are read by TMA (16-byte aligned base); beta and out are accessed
  // element-wise (2-byte alignment); the gate parameters as fp32 (4 bytes).
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (rows > 0) {
    const void* tma[] = {q, k, v, g};
    for (const void* p : tma)
      if (p == nullptr || !aligned16(p)) return KDA_ERR_INVALID_ARGUMENT;
    if (beta == nullptr || out == nullptr || !aligned(beta, 2) || !aligned(out, 2)) return KDA_ERR_INVALID_ARGUMENT;
  }
  // the chain kernel reads dt_bias four values at a time
  if (gate_here && (A_log == nullptr || dt_bias == nullptr || !aligned(A_log, 4) || !aligned16(dt_bias)))
    return KDA_ERR_INVALID_ARGUMENT;
  // states (FlashKDA README, "Kernel API"): each may be absent, bf16 or fp32, and two given
  // states share one dtype
  auto dtype_ok = [](kda_state_dtype d) { return d == KDA_STATE_BF16 || d == KDA_STATE_FP32; };
  if (initial_state != nullptr && (!dtype_ok(init_dtype) || !aligned16(initial_state))) return KDA_ERR_INVALID_ARGUMENT;
  if (final_state != nullptr && (!dtype_ok(final_dtype) || !aligned16(final_state))) return KDA_ERR_INVALID_ARGUMENT;
  if (initial_state == nullptr && init_dtype != KDA_STATE_NONE) return KDA_ERR_INVALID_ARGUMENT;
  if (final_state == nullptr && final_dtype != KDA_STATE_NONE) return KDA_ERR_INVALID_ARGUMENT;
  if (initial_state != nullptr && final_state != nullptr) {
    if (init_dtype != final_dtype) return KDA_ERR_INVALID_ARGUMENT;
    const size_t bytes = (size_t)s.N * s.H * s.V * s.K * (init_dtype == KDA_STATE_FP32 ? 4 : 2);
    const uintptr_t a = reinterpret_cast<uintptr_t>(initial_state), b = reinterpret_cast<uintptr_t>(final_state);
    if (a != b && a < b + bytes && b < a + bytes) return KDA_ERR_INVALID_ARGUMENT;   // partial overlap
  }
  DeviceInfo d;
  if (device_info(&d) != KDA_OK) return KDA_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return KDA_ERR_UNSUPPORTED_DEVICE;
  const kda_shape sc = chain_shape(s);
  const Layout L = make_layout(sc, d.sms);
  if (workspace == nullptr || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return KDA_ERR_WORKSPACE_TOO_SMALL;
  if (s.N == 0) return KDA_OK;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(ws + L.off_hdr);

  ScheduleParams sp;
  sp.cu_seqlens = cu_seqlens;
  sp.B = s.B;
  sp.T = s.T;
  sp.H = sc.H;
  sp.N = s.N;
  sp.seg_tokens = (int)L.seg_tokens;
  sp.seg_forced = forced_seg_tokens() != 0;
  sp.resident = 2 * (long long)std::max(d.sms, 1);
  sp.has_init = initial_state != nullptr;
  sp.has_final = final_state != nullptr;
  sp.hdr = hdr;
  sp.correct = reinterpret_cast<WorkItem*>(ws + L.off_correct);
  sp.forward = reinterpret_cast<WorkItem*>(ws + L.off_forward);
  sp.transition = reinterpret_cast<WorkItem*>(ws + L.off_transition);
  sp.cap_transition = L.cap_transition;
  sp.compose = reinterpret_cast<ComposeItem*>(ws + L.off_compose);
  sp.cap_correct = L.cap_correct;
  sp.cap_forward = L.cap_forward;
  sp.cap_compose = L.cap_compose;
  sp.cap_slots = L.cap_slots;
  sp.seg_rank = reinterpret_cast<int*>(ws + L.off_ranks);
  sp.cap_ranks = L.cap_ranks;
  sp.sm_arrivals = reinterpret_cast<int*>(ws + L.off_sm);
  int launches = 0;
  if (launch_schedule(sp, stream) != cudaSuccess) return KDA_ERR_CUDA;
  ++launches;
  mark(0, stream);

  ChainParams cp;
  std::memset(&cp, 0, sizeof(cp));
  if (rows > 0) {
    const bool v_ok = s.V == 64 ? encode_tile_map(&cp.tm_v, v, rows, s.H, 64)
                                : encode_halves_map(&cp.tm_v, v, rows, s.H, s.V);
    // K = 64: one 64-channel tile each of q, k and g
    const bool kg_ok = s.K == 64 ? encode_tile_map(&cp.tm_k, k, rows, s.H, 64) &&
                                       encode_tile_map(&cp.tm_g, g, rows, s.H, 64)
                                 : encode_halves_map(&cp.tm_k, k, rows, s.H) &&
                                       encode_halves_map(&cp.tm_g, g, rows, s.H);
    if (!encode_tile_map(&cp.tm_q, q, rows, s.H, s.K) || !kg_ok || !v_ok)
      return KDA_ERR_CUDA;
  }
  cp.beta = static_cast<const uint16_t*>(beta);
  cp.A_log = A_log;
  cp.dt_bias = dt_bias;
  cp.out = static_cast<uint16_t*>(out);
  cp.init_state = initial_state;
  cp.final_state = final_state;
  cp.ws_states = reinterpret_cast<float*>(ws + L.off_slots);
  cp.zero_flags = reinterpret_cast<int*>(ws + L.off_zero);
  cp.err = &hdr->err;
  cp.H = (int)s.H;
  cp.vsplit = (int)std::max<int64_t>(s.V / 128, 1);
  cp.vrows = s.V == 64 ? 64 : 128;
  cp.kdim = (int)s.K;
  cp.init_dtype = (int)init_dtype;
  cp.final_dtype = (int)final_dtype;
  cp.scale = scale;
  cp.lower_bound = lower_bound;
  cp.flags = (int)(flags & kValidFlags);
  // the state read as bf16 hi + lo where a gate may keep it (no decay fades the rounding
  // of a single bf16 copy): asked for, the safe gate near lower_bound 0, or a gate whose
  // decay the host cannot bound
  cp.precise = ((flags & KDA_PRECISE_STATE) != 0 || !uses_lower_bound(flags) || lower_bound > -0.25f) ? 1 : 0;
  cp.take = nullptr;
  cp.sm_arrivals = nullptr;

  // the transition runs of the split sequences' middle segments (a kernel of their own: the
  // forward runs' kernel carries none of their code); they usually stop after a few chunks
  // they usually stop after a few chunks: the forward launch overlaps them
  const bool transitions = L.cap_transition > 0;
  if (transitions) {
    cp.items = sp.transition;
    cp.item_count = &hdr->n_transition;
    if (launch_chain_aux(cp, (int)L.cap_transition, stream) != cudaSuccess) return KDA_ERR_CUDA;
    ++launches;
  }
  // every segment's forward run (outputs, local carries), longest first, two CTAs per SM
  // paired long with short
  cp.items = sp.forward;
  cp.item_count = &hdr->n_forward;
  cp.take = hdr->take;
  cp.sm_arrivals = sp.sm_arrivals;
  if (launch_chain(cp, (int)L.cap_forward, stream, transitions) != cudaSuccess) return KDA_ERR_CUDA;
  ++launches;
  mark(1, stream);
  if (L.cap_correct > 0) {
    ComposeParams cmp;
    cmp.ws_states = cp.ws_states;
    cmp.zero_flags = cp.zero_flags;
    cmp.items = sp.compose;
    cmp.item_count = &hdr->n_compose;
    if (launch_compose(cmp, (int)L.cap_compose, d.sms, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (L.cap_compose > 0) ++launches;
    // last launch: the corrections of segments 1 .. n-1 from their true entering states.  It
    // starts beside the composition: its runs set up and prepare their first chunks' operands
    // from the inputs, then wait for the composed states (so no profile mark between the two:
    // an event recorded there would order the launch after the composition)
    cp.items = sp.correct;
    cp.item_count = &hdr->n_correct;
    cp.take = nullptr;
    cp.sm_arrivals = nullptr;
    if (launch_chain_aux(cp, (int)L.cap_correct, stream, true) != cudaSuccess) return KDA_ERR_CUDA;
    ++launches;
  }
  mark(2, stream);
  mark(3, stream);
  t_last_launches = launches;
  return KDA_OK;
}

int kda_last_launch_count(void) { return t_last_launches; }

kda_status kda_set_profile_events(void* const* events, int n_events) {
  if (events == nullptr) {
    g_profile = false;
    return KDA_OK;
  }
  if (n_events != 4) return KDA_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < 4; ++i) g_profile_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_profile = true;
  return KDA_OK;
}

kda_status kda_check_device_error(const void* workspace, kda_stream_t stream_, int* flags) {
  if (workspace == nullptr || flags == nullptr) return KDA_ERR_INVALID_ARGUMENT;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  int err = 0;
  if (cudaMemcpy(&err, &static_cast<const WorkHeader*>(workspace)->err, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return KDA_ERR_CUDA;
  *flags = err;
  if (err & kErrTimeout) return KDA_ERR_TIMEOUT;
  if (err & kErrBadSeqlens) return KDA_ERR_BAD_SEQLENS;
  if (err & kErrGateRange) return KDA_ERR_GATE_RANGE;
  return KDA_OK;
}

kda_status kda_bwd_workspace_size(const kda_shape* shape, size_t* bytes) {
  if (bytes == nullptr) return KDA_ERR_INVALID_ARGUMENT;
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  if (shape->K != 128 || shape->V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  *bytes = std::max(make_bwd_layout(*shape).total, make_bwd_chunked_layout(*shape).total);
  return KDA_OK;
}

kda_status kda_bwd(const kda_shape* shape, const void* q, const void* k, const void* v, const void* g,
                   const void* beta, float scale, const float* A_log, const float* dt_bias, float lower_bound,
                   const void* initial_state, kda_state_dtype init_dtype, const int64_t* cu_seqlens,
                   const void* dout, const float* dfinal, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                   float* dh0, float* dA_log, float* ddt_bias, unsigned flags, void* workspace,
                   size_t workspace_bytes, kda_stream_t stream_) {
  kda_status st = check_shape(shape);
  if (st != KDA_OK) return st;
  const kda_shape s = *shape;
  if (s.K != 128 || s.V != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (cu_seqlens != nullptr && s.B != 1) return KDA_ERR_INVALID_ARGUMENT;
  if (cu_seqlens == nullptr && s.N != s.B) return KDA_ERR_INVALID_ARGUMENT;
  if ((long long)s.N * s.H * kBwdSlices > 0x7fffffffLL) return KDA_ERR_INVALID_ARGUMENT;
  if (!valid_flags(flags & ~(unsigned)KDA_BWD_RECURRENT)) return KDA_ERR_INVALID_ARGUMENT;
  const bool gate_here = !(flags & KDA_GATE_PREACTIVATED);
  if (uses_lower_bound(flags) && !(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_INVALID_ARGUMENT;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  // token tensors are read and written four (chunked form: eight) channels at a time
  if (s.B * s.T > 0) {
    const void* tok16[] = {q, k, v, g, dout, dq, dk, dv, dg};
    for (const void* p : tok16)
      if (p == nullptr || !aligned16(p)) return KDA_ERR_INVALID_ARGUMENT;
    if (beta == nullptr || dbeta == nullptr || !aligned(beta, 2) || !aligned(dbeta, 4))
      return KDA_ERR_INVALID_ARGUMENT;
  }
  if (gate_here && (A_log == nullptr || dt_bias == nullptr || !aligned(A_log, 4) || !aligned16(dt_bias)))
    return KDA_ERR_INVALID_ARGUMENT;
  if (initial_state != nullptr &&
      ((init_dtype != KDA_STATE_BF16 && init_dtype != KDA_STATE_FP32) || !aligned16(initial_state)))
    return KDA_ERR_INVALID_ARGUMENT;
  if (initial_state == nullptr && init_dtype != KDA_STATE_NONE) return KDA_ERR_INVALID_ARGUMENT;
  if ((dfinal != nullptr && !aligned16(dfinal)) || (dh0 != nullptr && !aligned16(dh0)) ||
      (dA_log != nullptr && !aligned(dA_log, 4)) || (ddt_bias != nullptr && !aligned(ddt_bias, 4)))
    return KDA_ERR_INVALID_ARGUMENT;
  // the gate with a lower bound takes the chunked form unless the recurrent one is asked for
  const bool chunked = uses_lower_bound(flags) && !(flags & KDA_BWD_RECURRENT);
  const BwdLayout L = make_bwd_layout(s);
  const BwdChunkedLayout C = make_bwd_chunked_layout(s);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return KDA_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < (chunked ? C.total : L.total)) return KDA_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo d;
  if (device_info(&d) != KDA_OK) return KDA_ERR_CUDA;
  if (d.major != 10 || d.minor != 3) return KDA_ERR_UNSUPPORTED_DEVICE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.g = static_cast<const uint16_t*>(g);
  p.beta = static_cast<const uint16_t*>(beta);
  p.dout = static_cast<const uint16_t*>(dout);
  p.dfinal = dfinal;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.init_state = initial_state;
  p.init_dtype = initial_state == nullptr ? 0 : (init_dtype == KDA_STATE_FP32 ? 2 : 1);
  p.cu = cu_seqlens;
  p.dq = dq;
  p.dk = dk;
  p.dg = dg;
  p.dv = dv;
  p.dbeta = dbeta;
  p.dh0 = dh0;
  p.dA_log = dA_log;
  p.ddt_bias = ddt_bias;
  p.T = s.T;
  p.BT = s.B * s.T;
  p.N = (int)s.N;
  p.H = (int)s.H;
  p.flags = (int)(flags & kValidFlags);
  p.scale = scale;
  p.lower_bound = lower_bound;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (chunked) {
    p.err = &reinterpret_cast<WorkHeader*>(ws + C.off_hdr)->err;
    p.items = reinterpret_cast<WorkItem*>(ws + C.off_items);
    p.item_count = &reinterpret_cast<WorkHeader*>(ws + C.off_hdr)->n_forward;
    p.citems = reinterpret_cast<WorkItem*>(ws + C.off_citems);
    p.citem_count = &reinterpret_cast<WorkHeader*>(ws + C.off_hdr)->n_correct;
    p.bslots = reinterpret_cast<float*>(ws + C.off_bslots);
    // cut each sequence into parts when the chains alone would leave most SMs idle: the most parts
    // (kBwdMaxParts, halving) that keep the 2 parts runs per (sequence, head) within one wave of
    // two CTAs per SM
    const int64_t NH = s.N * s.H, wave = 2 * (int64_t)std::max(d.sms, 1);
    p.parts = 1;
    if (NH <= kBwdMaxSplitChains)
      for (int P = kBwdMaxParts; P > 1; P /= 2)
        if (2 * P * NH <= wave) {
          p.parts = P;
          break;
        }
    p.s0 = reinterpret_cast<const uint16_t*>(ws + C.off_s0);
    p.ds1 = reinterpret_cast<const uint16_t*>(ws + C.off_ds1);
    p.vn = reinterpret_cast<const float*>(ws + C.off_vn);
    p.dvn = reinterpret_cast<const float*>(ws + C.off_dvn);
    p.xp = reinterpret_cast<float*>(ws + C.off_xp);
    p.zs = reinterpret_cast<float*>(ws + C.off_zs);
    p.ppart = reinterpret_cast<float*>(ws + C.off_ppart);
    p.nblk = C.nblk;
    p.nslots = C.nslots;
    p.sms = std::max(d.sms, 1);
    // the chains: per part of each (sequence, head) a forward run storing S0 and Vn and a reverse
    // run storing dS1 and dVn
    ChainParams cp;
    std::memset(&cp, 0, sizeof(cp));
    const int64_t rows = s.B * s.T;
    if (rows > 0) {
      if (!encode_tile_map(&cp.tm_q, q, rows, s.H) || !encode_halves_map(&cp.tm_k, k, rows, s.H) ||
          !encode_halves_map(&cp.tm_g, g, rows, s.H) || !encode_halves_map(&cp.tm_v, v, rows, s.H) ||
          !encode_halves_map(&cp.tm_dout, dout, rows, s.H))
        return KDA_ERR_CUDA;
    }
    cp.beta = p.beta;
    cp.A_log = A_log;
    cp.dt_bias = dt_bias;
    cp.init_state = initial_state;
    cp.init_dtype = p.init_dtype;
    cp.dfinal = dfinal;
    cp.dh0 = dh0;
    cp.save_s0 = reinterpret_cast<uint16_t*>(ws + C.off_s0);
    cp.save_ds1 = reinterpret_cast<uint16_t*>(ws + C.off_ds1);
    cp.save_vn = reinterpret_cast<float*>(ws + C.off_vn);
    cp.save_dvn = reinterpret_cast<float*>(ws + C.off_dvn);
    cp.items = p.items;
    cp.item_count = p.item_count;
    cp.ws_states = p.bslots;
    cp.err = p.err;
    cp.H = (int)s.H;
    cp.vsplit = 1;
    cp.kdim = 128;
    cp.vrows = 128;
    cp.scale = scale;
    cp.lower_bound = lower_bound;
    cp.flags = (int)(flags & kValidFlags);
    cp.precise = 0;
    // profile marks: the runs, the chains, the state products, the chunk gradients
    if (launch_bwd_chunked(p, 0, stream) != cudaSuccess) return KDA_ERR_CUDA;
    mark(0, stream);
    if (launch_chain_bwd(cp, (int)(2 * p.parts * NH), stream) != cudaSuccess) return KDA_ERR_CUDA;
    for (int l = 1; l < p.parts; ++l) {   // the corrections of the cut sequences, cut by cut
      ChainParams cc = cp;
      cc.items = p.citems + (size_t)(l - 1) * 2 * NH;
      cc.item_count = p.citem_count;
      if (launch_chain_bwd(cc, (int)(2 * NH), stream, true) != cudaSuccess) return KDA_ERR_CUDA;
    }
    mark(1, stream);
    if (launch_bwd_chunked(p, 2, stream) != cudaSuccess) return KDA_ERR_CUDA;
    mark(2, stream);
    if (launch_bwd_chunked(p, 3, stream) != cudaSuccess) return KDA_ERR_CUDA;
    mark(3, stream);
    const bool work = p.BT > 0 && p.H > 0;
    t_last_launches = 1 + (s.N > 0 ? p.parts : 0) + (work ? 2 : 0) +
                      ((dA_log == nullptr && ddt_bias == nullptr) ? 0 : (C.nblk > 0 ? 2 : 1));
    return KDA_OK;
  }
  p.prep = reinterpret_cast<float*>(ws + L.off_prep);
  p.ckpt = reinterpret_cast<float*>(ws + L.off_ckpt);
  p.part = reinterpret_cast<float*>(ws + L.off_part);
  p.dA_tok = reinterpret_cast<float*>(ws + L.off_dA);
  p.ppart = reinterpret_cast<float*>(ws + L.off_ppart);
  p.err = &reinterpret_cast<WorkHeader*>(ws + L.off_hdr)->err;
  p.nblk = L.nblk;
  // profile marks after each phase: prep, stored-state forward, reverse, chain rule
  for (int phase = 0; phase < 4; ++phase) {
    if (launch_bwd(p, phase, stream) != cudaSuccess) return KDA_ERR_CUDA;
    mark(phase, stream);
  }
  t_last_launches = (p.BT * p.H > 0 ? 2 : 0) + (p.N > 0 ? 2 : 0) +
                    ((flags & KDA_GATE_PREACTIVATED) || (dA_log == nullptr && ddt_bias == nullptr)
                         ? 0 : (L.nblk > 0 ? 2 : 1));
  return KDA_OK;
}

}  // extern "C"
