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
// Register split (setmaxnreg): the kernel is launched with kFmhaLaunchRegs per thread; the
// softmax warpgroups grow to kSoftmaxRegs, the TMA/MMA warpgroup shrinks to kControlRegs.
// The split must not exceed the launch total: 2*128*224 + 128*56 = 384*168.
constexpr int kFmhaLaunchRegs = 168;
constexpr int kSoftmaxRegs = 224;
constexpr int kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kFmhaThreads * kFmhaLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kMaxL = 1 << 24;        // positions and row indices stay exact in FP32 / int32

// Bits of the device error word.
constexpr int kErrProducer = 1;       // TMA warp gave up on a wait
constexpr int kErrMma = 2;            // MMA warp gave up on a wait
constexpr int kErrSoftmax = 4;        // softmax / epilogue warps gave up on a wait

// RoPE pre-pass: rotate q and k (all planes) in FP32 and cast back to the storage dtype.
struct RopeArgs {
  const uint16_t* q;
  const uint16_t* k;
  uint16_t* q_out;
  uint16_t* k_out;
  const int32_t* positions;   // [L] or nullptr for 0..L-1
  long long planes;           // B * H * nmaps rows-of-L planes in q (and in k)
  int L;
  int planes_per_block;
  float inv_freq[kHeadDim / 2];
};

// Attention kernel arguments (tensor maps are passed separately as __grid_constant__).
struct FmhaArgs {
  void* out;                  // [B, H, L, d_v]
  int* err;                   // device error word (bits above), atomically OR-ed
  int L;
  int H;
  int n_qblocks;              // CTAs per (b, h)
  int window;                 // < 0: full attention, else |i - j| <= window (< L - 1)
  float scale_log2;           // log2(e) / sqrt(d)
  unsigned long long timeout_ns;
  float lambda[kMaxDiffHeads];
};

// Rows of queries one CTA owns: two 128-row tiles (standard) or one tile with two maps.
constexpr int fmha_rows_per_cta(bool diff) { return diff ? kBlockM : 2 * kBlockM; }

// Blocks of the RoPE kernel resident per SM (from the occupancy calculator).
int rope_blocks_per_sm();
cudaError_t rope_launch(const RopeArgs& a, bool bf16, int num_sms, int blocks_per_sm, cudaStream_t stream);

cudaError_t fmha_set_attributes();
// Registers per thread ptxas assigned to each attention kernel (must equal kFmhaLaunchRegs).
bool fmha_check_registers(int* got);
cudaError_t fmha_launch(bool diff, bool bf16, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v, const FmhaArgs& a, long long num_ctas,
                        cudaStream_t stream);

// Library-internal hooks defined in sa_api.cu (not part of the exported C ABI).
sa_status set_error(sa_status st, const char* msg);
int handle_device(sa_attn_t h);
sa_status rope_attn_into(const char* fn, sa_attn_t h, const void* q, const void* k, const void* v,
                         const int32_t* positions, void* out, int B, int H, int L, int d,
                         int window, const float* lambda, sa_dtype dtype, void* q_rot, void* k_rot,
                         sa_stream_t stream);

}  // namespace sa
