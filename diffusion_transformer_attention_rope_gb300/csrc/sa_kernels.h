// sa_kernels.h -- host-side view of the two kernels of the RoPE + attention core:
// argument structs, tile constants and launchers.  No torch types anywhere.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sa_attn.h"

namespace sa {

constexpr int kHeadDim = 64;          // d of q and k (the only supported value)
constexpr int kBlockM = 128;          // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;          // keys per K/V tile
constexpr int kMaxDiffHeads = 128;    // lambda is carried by value in the kernel arguments
constexpr int kFmhaThreads = 384;     // 3 warpgroups: 2 softmax + (2 TMA producers, 2 MMA issuers)
// Register split (setmaxnreg) of the standard kernel: it is launched with kFmhaLaunchRegs per
// thread; the softmax warpgroups grow to kSoftmaxRegs, the TMA/MMA warpgroup shrinks to
// kControlRegs (ptxas allocates each region within its new count).  The split must not exceed
// the launch total: 2*128*224 + 128*56 = 384*168.  The differential kernel runs without a split:
// its softmax fits the launch registers and its control warps then need no spills (measured
// 3% faster at L = 4096); the standard kernel's softmax needs the grow.
constexpr int kFmhaLaunchRegs = 168;
constexpr int kSoftmaxRegs = 224;
constexpr int kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kFmhaThreads * kFmhaLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kMaxL = 1 << 24;        // positions and row indices stay exact in FP32 / int32
constexpr int kHostChunks = 4;        // sa_rope_attn_host: planes are copied and computed in chunks

// Bits of the device error word.
constexpr int kErrProducer = 1;       // TMA warp gave up on a wait
constexpr int kErrMma = 2;            // MMA warp gave up on a wait
constexpr int kErrSoftmax = 4;        // softmax / epilogue warps gave up on a wait

// RoPE pre-pass: rotate q and k (all planes) in FP32 and cast back to the storage dtype.
struct RopeArgs {
  const uint16_t* q;          // nullptr: k only (the attention kernel rotates q)
  const uint16_t* k;
  uint16_t* q_out;
  uint16_t* k_out;
  float2* cs;                 // nullptr, or [L][32] (cos, sin) pairs written for the Q prologue
  const int32_t* positions;   // [L] or nullptr for 0..L-1
  long long planes;           // B * H * nmaps rows-of-L planes in q (and in k)
  int L;
  int planes_per_block;
  float inv_freq[kHeadDim / 2];
  // QK-RMSNorm before the rotation (qk_norm != 0): x * gamma / sqrt(mean(x^2) + eps) per row
  int qk_norm;
  float eps;
  float gamma_q[kHeadDim];
  float gamma_k[kHeadDim];
};

// Attention kernel arguments (tensor maps are passed separately as __grid_constant__).
//
// Grid.  A unit is the query rows of one (batch, head) block (fmha_rows_per_cta) with the key
// tiles they visit.  CTAs [0, whole_ctas) take units 0 .. whole_ctas - 1 whole.  When the
// units do not fill the last wave of the GPU, the units after those (the tail) are each cut
// into tail_k pieces of their key range, one CTA per piece, so that the last wave is spread
// over more SMs; a piece stores its un-normalised O, running max and row sum (FP32) in
// `partials` and the piece that finishes last merges them and writes the output.
struct FmhaArgs {
  void* out;                  // [B, H, L, d_v]
  int* err;                   // device error word (bits above), atomically OR-ed
  int L;
  int H;
  int n_qblocks;              // units per (b, h)
  int window;                 // < 0: full attention, else |i - j| <= window (< L - 1)
  float scale_log2;           // log2(e) / sqrt(d)
  int whole_ctas;             // CTAs that take a whole unit (the first ones)
  int tail_k;                 // pieces per tail unit (1: no pieces)
  int wave;                   // CTAs resident at once (one per SM): the Q-prefetch distance
  unsigned epoch;             // nonzero, distinct for every launch (tags the unit counters)
  const float2* cs;           // nullptr: q is already rotated; else q is raw and is rotated in the
                              // prologue with this [L][32] (cos, sin) table of the RoPE pass
  unsigned long long* counters;  // tail_k > 1: [units] epoch-tagged piece counts
  float* partials;            // tail_k > 1: one slot of fmha_partial_floats per piece CTA
  unsigned long long timeout_ns;
  float lambda[kMaxDiffHeads];
  // Q prologue only (cs != nullptr): QK-RMSNorm of each raw q row before its rotation
  int qk_norm;
  float eps;
  float gamma_q[kHeadDim];
  // the table's row stride in float4 units per pair group (L for a per-call table, the
  // capacity for the handle's table of positions 0 .. capacity - 1)
  int cs_stride;
  // cs is the handle's table, written when the handle was created: the prologue needs nothing
  // from the RoPE pass
  int cs_static;
};

// Rows of queries in one unit: two 128-row tiles (standard) or one tile with two maps.
constexpr int fmha_rows_per_cta(bool diff) { return diff ? kBlockM : 2 * kBlockM; }
// FP32 values of one partial-result slot: per stream (tile or map) and row, O (d_v values),
// then the running max and the row sum.
constexpr int fmha_partial_floats(bool diff) { return 2 * kBlockM * ((diff ? 2 * kHeadDim : kHeadDim) + 2); }
// Most piece CTAs one launch uses (the split workspace is sized for that many slots), and most
// pieces one unit is cut into.
constexpr int kMaxPieces = 160;
constexpr int kMaxTailK = 4;

// Blocks of the RoPE kernel resident per SM (from the occupancy calculator) for the variant
// that rotates q as well as k (or k only), without or with the QK-RMSNorm.
int rope_blocks_per_sm(bool with_q, bool qk_norm);
cudaError_t rope_launch(const RopeArgs& a, bool bf16, int num_sms, int blocks_per_sm, cudaStream_t stream);
// The k-only pass (no table) as at most `blocks` blocks of kRopeSideThreads that walk the
// pass's items: for a call whose attention grid leaves SMs idle, the pass then occupies at
// most `blocks` SMs and the attention CTAs start on the others at once.
constexpr int kRopeSideThreads = 512;
cudaError_t rope_side_launch(const RopeArgs& a, bool bf16, int blocks, cudaStream_t stream);
// The (cos, sin) table alone (a.cs, [16][a.L] float4), with the pass's arithmetic.
cudaError_t rope_table_launch(const RopeArgs& a, cudaStream_t stream);

// FP32-input path (sa_tf32.cu): RoPE of q and k in FP32, results rounded to TF32.
struct RopeF32Args {
  const float* q;
  const float* k;
  float* q_out;
  float* k_out;
  const int32_t* positions;   // [L] or nullptr for 0..L-1
  long long planes;           // B * H * 2 planes of L rows in q (and in k)
  int L;
  float inv_freq[kHeadDim / 2];
  // v [planes_v][L][128] -> v_t [planes_v][128][L_pad] (TF32), or v == nullptr: no transpose
  const float* v;
  float* v_t;
  long long planes_v;
  int L_pad;                  // L rounded up to a multiple of 4 (16-byte rows)
};

// FP32-input differential attention (TF32 products): one CTA per (batch, head, 128-row block).
struct FmhaF32Args {
  float* out;                 // [B, H, L, 128]
  int* err;
  int L;
  int H;
  int n_qblocks;
  int window;                 // < 0: full attention
  float scale_log2;
  unsigned long long timeout_ns;
  float lambda[kMaxDiffHeads];
};

cudaError_t rope_f32_launch(const RopeF32Args& a, int num_sms, cudaStream_t stream);
cudaError_t fmha_tf32_set_attributes();
// false when the kernel's binary is not sm_103a code
bool fmha_tf32_check(int* regs);
cudaError_t fmha_tf32_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FmhaF32Args& a, long long num_ctas, cudaStream_t stream);

// Differential attention with a narrow window (sa_swa.cu): one CTA per SM walks a contiguous
// run of 128-row query blocks (units); raw q is rotated in its prologue with the (cos, sin) table
// (or taken as rotated already).
constexpr int kSwaMaxWindow = 256;    // windows up to this width take this kernel (measured faster
                                      // than the general one at 17 and 256, slower without a window)
struct FmhaSwaArgs {
  void* out;                  // [B, H, L, 128]
  int* err;
  int L;
  int H;
  int n_qblocks;              // 128-row blocks per (batch, head)
  int window;                 // 0 <= window <= kSwaMaxWindow
  float scale_log2;
  unsigned long long timeout_ns;
  long long units;            // B * H * n_qblocks
  const float2* cs;           // [16][cs_stride] float4 (cos, sin) table, or nullptr: q rotated already
  int cs_stride;
  int cs_static;              // the handle's table (no wait for the RoPE pass)
  float lambda[kMaxDiffHeads];
  // QK-RMSNorm of each raw q row in the prologue (cs != nullptr only)
  int qk_norm;
  float eps;
  float gamma_q[kHeadDim];
};

cudaError_t fmha_swa_set_attributes();
bool fmha_swa_check();
// to: the output [B*H][L][128] (box 64 x 32 rows), written by the epilogue's TMA stores
cudaError_t fmha_swa_launch(bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const FmhaSwaArgs& a, int num_ctas, cudaStream_t stream);

cudaError_t fmha_set_attributes();
// Registers per thread ptxas assigned to each attention kernel (must equal kFmhaLaunchRegs);
// false also when a kernel's binary is not sm_103a code.
bool fmha_check_registers(int* got);
cudaError_t fmha_launch(bool diff, bool bf16, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, const FmhaArgs& a, long long num_ctas,
                        cudaStream_t stream);

// Library-internal hooks defined in sa_api.cu (not part of the exported C ABI).
sa_status set_error(sa_status st, const char* msg);
int handle_device(sa_attn_t h);
// The handle's slot for the noalloc scratch address (nullptr until its first noalloc call).
void** handle_noalloc_slot(sa_attn_t h);
// The shape, dtype and lambda checks of sa_rope_attn, in its order.
sa_status check_call(const char* fn, int B, int H, int L, int d, const float* lambda, sa_dtype dtype);
sa_status rope_attn_into(const char* fn, sa_attn_t h, const void* q, const void* k, const void* v,
                         const int32_t* positions, void* out, int B, int H, int L, int d,
                         int window, const float* lambda, sa_dtype dtype, void* q_rot, void* k_rot,
                         sa_stream_t stream);

}  // namespace sa
