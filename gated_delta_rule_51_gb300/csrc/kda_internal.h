// kda_internal.h -- shared definitions between the host launcher and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kChunk = 16;   // tokens per chunk
constexpr int kDimK = 128;
constexpr int kDimV = 128;

// One unit of sequential work: a run of chunks of one (sequence, head).
//   kModeForward     outputs written, state carried from in_slot to out_slot
//   kModeCorrect     v taken as zero: propagates the difference D between a segment's true
//                    entering state and the zero state its forward run started from; adds
//                    scale * q^T D to the outputs that run wrote and stops once D is exactly
//                    zero in fp32 (it then stays zero)
//   kModeTransition  v taken as zero from the identity: the segment's transition matrix,
//                    stopped (and flagged zero) once it is exactly zero in fp32
//   kModeReverse     (backward chains only) the state gradient dS carried from the sequence's
//                    end to its start: dout in place of v, chunks last first, dS_0 written out
//   kModeReverseCorrect (backward, split sequences) the reverse run with dout taken as zero from
//                    the true dS at a segment's end, adding to what the segment's reverse run
//                    stored; kModeCorrect does the same for the forward runs (v taken as zero)
enum : int { kModeForward = 0, kModeCorrect = 1, kModeTransition = 2, kModeReverse = 3, kModeReverseCorrect = 4 };
// in_slot values below zero:
enum : int { kInZero = -1, kInIdentity = -2, kInUser = -3 };
// out_slot values below zero:
enum : int { kOutNone = -1, kOutUser = -3 };

struct WorkItem {
  int row0;      // first token row in the flattened [B*T] token index
  int len;       // tokens in this run (may be 0)
  int head;
  int mode;      // kModeForward / kModeCorrect / kModeTransition
  int seq;       // sequence index n (user state row)
  int in_slot;   // initial state source
  int out_slot;  // final state target
  int aux_slot;  // kModeCorrect with a final state: the slot holding the segment's local final
                 // state (from zero), which the run's own final difference is added to
};

// Device-side work list built by the scheduling kernel inside the workspace.
struct WorkHeader {
  int err;             // error word (bit flags, see kda_device.cuh)
  int n_correct;       // number of correction items (the last phase)
  int n_forward;       // number of forward runs (the first chain launch)
  int n_compose;       // number of (sequence, head) carry chains to compose
  int take[3];         // forward runs handed out: total, from the head, from the tail
  int n_transition;    // number of transition runs (their own launch, before the forward runs)
};
constexpr int kMaxSmIds = 256;   // per-SM arrival counters of the forward launch

struct ComposeItem {
  int head;
  int first_q_slot;   // workspace slot holding the true state after segment 0
  int first_p_slot;   // slot of the transition of segment 1 (P_1)
  int n_steps;        // number of compositions (segments 1 .. n_seg-2)
  // step s (1 <= s <= n_steps) uses P slot first_p_slot + (s-1) and Q slots
  // first_q_slot + s - 1 (input) and first_q_slot + s (carry, overwritten); a P slot
  // flagged zero (ComposeParams::zero_flags) is neither read nor multiplied
};

struct ChainParams {
  CUtensorMap tm_q;                  // 3-D map over [B*T, H, 128] bf16, box {64, 1, 16}
  CUtensorMap tm_k, tm_g, tm_v;      // 4-D maps {64, H, B*T, 2 halves (v: 2 V/128)}, box {64, 1, 16, 2}
  const uint16_t* beta;                // [B*T, H] bf16 logits
  const float* A_log;                  // [H]
  const float* dt_bias;                // [H, 128]
  uint16_t* out;                       // [B*T, H, 128] bf16
  const void* init_state;              // [N, H, 128, 128] or null
  void* final_state;                   // [N, H, 128, 128] or null
  float* ws_states;                    // workspace state slots, 128*128 fp32 each
  int* zero_flags;                     // per slot: 1 when a transition run found it exactly zero
  const WorkItem* items;
  const int* item_count;
  int* take;                           // non-null: CTAs pick items by SM pairing (WorkHeader::take)
  int* sm_arrivals;                    // [kMaxSmIds] CTAs that started on each SM
  int* err;
  int H;
  int init_dtype;                      // kda_state_dtype
  int final_dtype;
  float scale;
  float lower_bound;
  int flags;                           // kGatePreactivated | kBetaPreactivated | kNoQkL2Norm | kGateSoftplus
  int vsplit;                          // V / 128: work-item heads are (head, 128-column value block)
  int kdim;                            // K: 128, or 64 (channels 64-127 then run as zeros)
  int vrows;                           // value rows a chain carries to the caller: 128, or 64 for V = 64
                                       // (rows 64-127 then stay zero: v's second 64 columns read as 0)
  int precise;                         // 1: the precise-state kernels (state, W read as bf16 hi + lo)
  // Backward chains (kChainBwd kernels) only.  Per (chunk slot, head), slot = seq + row0 / 16 +
  // chunk (unique across sequences): the forward runs store each chunk's entering state (the
  // bf16 copy of S^T, piece-major: 16-byte piece q of row v at [q][v]) and Vn ([16 tokens][128 v]
  // fp32); the reverse runs the gradient dS_1 at each chunk's end and dVn, in the same layouts.
  CUtensorMap tm_dout;                 // 4-D map over dout, as tm_v
  uint16_t* save_s0;
  float* save_vn;
  uint16_t* save_ds1;
  float* save_dvn;
  const float* dfinal;                 // reverse runs: dS at the sequence's end, fp32 [N, H, 128, 128], or null
  float* dh0;                          // reverse runs: dS at its start (fp32), or null
};

struct ComposeParams {
  float* ws_states;
  const int* zero_flags;
  const ComposeItem* items;
  const int* item_count;
};

struct ScheduleParams {
  const int64_t* cu_seqlens;  // null: fixed-length rows of T tokens
  int64_t B, T, H, N;
  int seg_tokens;             // maximum tokens per segment (multiple of 16)
  int seg_forced;             // seg_tokens was set by the caller: split at it, whatever the lengths
  long long resident;         // chain CTAs resident on the device at once
  int has_init;
  int has_final;
  WorkHeader* hdr;
  WorkItem* correct;
  WorkItem* forward;
  WorkItem* transition;
  ComposeItem* compose;
  long long cap_correct, cap_forward, cap_transition, cap_compose, cap_slots;
  int* seg_rank;              // scratch: position of each forward run's segment in the list
  long long cap_ranks;
  int* sm_arrivals;           // [kMaxSmIds], zeroed here for the forward launch
};

// Steps the caller already did (include/kda.h KDA_GATE_PREACTIVATED, ...).
constexpr int kGatePreactivated = 1;
constexpr int kBetaPreactivated = 2;
constexpr int kNoQkL2Norm = 4;
constexpr int kGateSoftplus = 8;   // ghat = -exp(A_log) softplus(g + dt_bias), no lower bound
constexpr unsigned kValidFlags = 15;
// chain-kernel variant bits (not caller flags): K = 64 or V = 64, the padded shapes; and the
// precise-state kernels (one CTA per SM)
constexpr int kChainPadded = 16;
constexpr int kChainPrecise = 32;
constexpr int kChainBwd = 64;   // the backward's chains: storing forward runs and reverse runs
constexpr int kChainAux = 128;  // the correction and transition runs' kernels (the others carry none of their code)

struct DecodeParams {
  const uint16_t *q, *k, *v, *g, *beta;  // bf16 [B, T, H, K] (v [B, T, H, V]; beta [B, T, H], logits)
  uint16_t* out;                          // bf16 [B, T, H, V]
  const float* A_log;                     // [H]
  const float* dt_bias;                   // [H, K]
  void* state;                            // [B, H, V, K], read and written in place
  int state_dtype;                        // 1 bf16, 2 fp32
  int vsplit;                             // V / 64: 64-row CTAs per (sequence, head)
  int kdim;                               // K: 128, or 64 (channels 64-127 then run as zeros)
  int flags;                              // kGatePreactivated | kBetaPreactivated | kNoQkL2Norm | kGateSoftplus
  int B, T, H;
  float scale, lower_bound;
};

// The backward pass (kda_bwd.cu): K = V = 128.
struct BwdParams {
  const uint16_t *q, *k, *v, *g, *beta;   // bf16 inputs of the forward ([B, T, H, 128]; beta [B, T, H])
  const uint16_t* dout;                   // bf16 [B, T, H, 128]: dL/d out
  const float* dfinal;                    // fp32 [N, H, 128, 128]: dL/d final_state, or null
  const float* A_log;                     // [H]
  const float* dt_bias;                   // [H, 128]
  const void* init_state;                 // [N, H, 128, 128] of init_dtype, or null
  int init_dtype;                         // 0 none, 1 bf16, 2 fp32
  const int64_t* cu;                      // [N + 1] or null
  float *dq, *dk, *dg, *dv, *dbeta;       // fp32 gradients ([B, T, H, 128]; dbeta [B, T, H])
  float* dh0;                             // fp32 [N, H, 128, 128] or null
  float *dA_log, *ddt_bias;               // fp32 [H], [H, 128] or null
  float* prep;                            // workspace: per token-head alpha, kh, qh, beta, rq, rk
  float* ckpt;                            // workspace: the state every kBwdChunk tokens
  float* part;                            // workspace: per row-slice partial dqh, dkh, dalpha, dbeta
  float* dA_tok;                          // workspace: per token-head dA_log terms
  float* ppart;                           // workspace: per token-block parameter sums
  int* err;                               // error word (kErrBadSeqlens)
  int64_t T;                              // tokens per sequence (cu == null) or the total
  int64_t BT;                             // B * T
  int N, H, flags, nblk;
  float scale, lower_bound;
  // The chunked path (kda_bwd.cu, kBwdChunked*): per (chunk slot, head), slot = n + row0(n) / 16 + c,
  // what the backward chains stored, and the state products of the chunk.
  const uint16_t* s0;                     // [slot][H] bf16 copies of S^T entering the chunk, piece-major:
                                          // columns 8 q .. 8 q + 7 of row v at [q][v][8]
  const float* vn;                        // [slot][H][16][128]: Vn
  const uint16_t* ds1;                    // dS at the chunk's end, as s0
  const float* dvn;                       // dVn, as vn
  float* xp;                              // [slot][H][3][16][128]: dO S0^T, Vn dS1^T, dVn S0^T
  float* zs;                              // [slot][H][128]: sum over v of dS1 * S0
  WorkItem* items;                        // the chains' runs: 2 parts per (sequence, head)
  int* item_count;
  WorkItem* citems;                       // the correction runs of split sequences: parts - 1 launches,
                                          // two per (sequence, head) each
  int* citem_count;
  float* bslots;                          // 2 parts - 1 128 x 128 fp32 states per (sequence, head)
  int parts;                              // cut each sequence into up to this many parts (1 or 2)
  int64_t nslots;
  int sms;                                // the device's SM count (persistent CTAs: two per SM)
};

// Backward workspace regions, in floats per unit.
constexpr int kBwdChunk = 8;              // tokens between two stored states
constexpr int kBwdRowStride = 388;        // floats per token-head in prep and part (128 x 3 + 4)
constexpr int kBwdSlices = 4;             // row slices (CTAs) per head in the recurrences
constexpr int kBwdParamTokens = 256;      // tokens per block of the parameter reduction
// The chunked backward's chains: parts per sequence at most.  Four parts measured slower than two
// on the fixed batch (chains 0.48 against 0.39 ms): their three correction launches run one after
// another, each for the tens of chunks its state takes to decay to exactly zero.
constexpr int kBwdMaxParts = 2;
constexpr int kBwdMaxSplitChains = 256;  // (sequence, head) chains beyond which no sequence is cut
constexpr int kBwdParamStride = 132;      // floats per (block, head): 128 ddt_bias + dA_log + pad

// Host-side launchers (defined in the .cu files).
cudaError_t launch_schedule(const ScheduleParams& p, cudaStream_t s);
// overlap_prev: the launch may start while the stream's previous kernel still runs (programmatic
// dependent launch); its CTAs wait for that kernel's completion before they exit
cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev = false);
cudaError_t launch_chain_precise(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev = false);
cudaError_t launch_chain_bwd(const ChainParams& p, int grid, cudaStream_t s, bool corrections = false);
// overlap_prev: launched to start beside the previous kernel of the stream (programmatic
// dependent launch); the runs wait for it before they read a state slot or touch the outputs
cudaError_t launch_chain_aux(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev = false);
cudaError_t launch_compose(const ComposeParams& p, int grid, int sms, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s);
// phases 0-3: prep, stored-state forward, reverse, chain rule and parameter sums
cudaError_t launch_bwd(const BwdParams& p, int phase, cudaStream_t s);
// the chunked path around the chains' launch (launch_chain_bwd): phase 0 the error word and the
// runs; 2 the state products; 3 the chunk gradients and the parameter sums
cudaError_t launch_bwd_chunked(const BwdParams& p, int phase, cudaStream_t s);

}  // namespace kda
