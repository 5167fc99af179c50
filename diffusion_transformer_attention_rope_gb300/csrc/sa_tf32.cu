// sa_tf32.cu -- the FP32-input form of SAME-L's differential sliding-window attention for
// sm_103a (GB300): RoPE of q and k in FP32, then
//   out = softmax(q1' k1'^T / sqrt(d)) v - lambda_h * softmax(q2' k2'^T / sqrt(d)) v
// with both attention products on the tensor cores in TF32 (FP32 accumulate), the softmax in
// FP32 and the subtraction in FP32 on the FP32 accumulators, and the optional symmetric window
// |i - j| <= w.  HF discussion #6 "sm_120 SAME-L": the decoder's attention projections are FP32
// islands, and the shipped kernel runs both attention products as TF32 MMAs with FP32
// accumulation ("How the kernels differ"); the window is the "Three gotchas" one.
//
// Two kernels:
//   rope_f32_kernel   q', k' = RoPE(q), RoPE(k) in FP32 (the 16-bit pass's angle and sin/cos
//                     arithmetic), each value then rounded to TF32 (to nearest, ties away), the
//                     precision the products use; and v transposed to v^T [d_v][L] (keys
//                     contiguous, rows padded to a multiple of 4 keys), rounded the same way.
//                     kind::tf32 MMAs take K-major operands only (an MN-major B operand gives
//                     zeros, measured on GB300), so the P.V product reads v^T.
//   fmha_tf32_kernel  one CTA per (batch, head, 128-row query block), both maps: 384 threads =
//                     softmax warpgroup per map (thread = query row = TMEM lane), a control
//                     warpgroup (warp 8: TMA of Q and the K ring; warp 9: TMEM allocation and
//                     the MMA issuer of map 0; warp 10: the MMA issuer of map 1; warp 11: TMA
//                     of the V ring).  Key tiles of 64 keys; per tile and map:
//                       S = Q K^T       kind::tf32, A and B K-major 128-byte-swizzled smem
//                       P = exp2(S c - m)  softmax warps: reducing load of S (row max), lazy
//                                      rescale of O (running max grows by more than 2^8),
//                                      FP32 exponentials and row sum, P rounded to TF32 and
//                                      stored over S in tensor memory
//                       O += P V        kind::tf32, A = P from tensor memory, B = v^T K-major
//                     S is double-buffered per map, so the next S MMA overlaps the softmax.
// Tensor memory (512 columns): map m at 256 m: S buffer 0 | S buffer 1 | O = 64 | 64 | 128.
// Shared memory: Q 64 KB (2 maps x 2 atoms of 32 dims), K ring 2 x 32 KB, v^T ring 2 x 32 KB
// (128 values x 2 atoms of 32 keys).  A window's first key is rounded down to a multiple of 4, so
// that the v^T copies start on a 16-byte boundary.
// Every wait is bounded as in the 16-bit kernels.
#include <cuda.h>

#include "sa_kernels.h"
#include "sa_pipe.cuh"
#include "sa_ptx.cuh"

namespace sa {
namespace {

// ------------------------------------------------------------------------------ RoPE, FP32

constexpr int kRopeF32Rows = 32;       // positions per block
constexpr int kRopeF32Threads = 128;   // 32 positions x 4 groups of 8 rotation pairs

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_f4(float* p, float4 v) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Rotate 8 rotate-half pairs of one FP32 row: lo = x[8g .. 8g+8), hi = x[32+8g .. 32+8g+8),
// with the pass's arithmetic (the 16-bit pass's rope_rotate8 without its cast), then round each
// result to TF32.
__device__ __forceinline__ void rope_rotate8_f32(float (&lo)[8], float (&hi)[8], const float (&c)[8],
                                                 const float (&s)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = lo[i], b = hi[i];
    lo[i] = round_tf32(fmaf(a, c[i], -(b * s[i])));
    hi[i] = round_tf32(fmaf(b, c[i], a * s[i]));
  }
}

// v^T of keys [l0, l0 + 32) of v plane pl: the rows v[l][0 .. 128) read as float4 per lane,
// staged in shared memory, written as 128 rows of 32 keys (TF32) of v^T [128][L_pad] (keys past
// L as zeros).  Every thread of the block takes part (two block barriers).
__device__ __forceinline__ void transpose_v_item(const RopeF32Args& a, int l0, long long pl,
                                                 float (*tile)[kRopeF32Rows + 1]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* src = a.v + static_cast<size_t>(pl) * a.L * (2 * kHeadDim);
  float* dst = a.v_t + static_cast<size_t>(pl) * (2 * kHeadDim) * a.L_pad;
  // row l0 + 4 j + warp: each lane loads 4 consecutive values of the row's 128 (all 8 loads
  // issued before the first use)
  float4 x[kRopeF32Rows / 4];
#pragma unroll
  for (int j = 0; j < kRopeF32Rows / 4; ++j) {
    const int l = l0 + 4 * j + warp;
    x[j] = l < a.L ? ld_stream_f4(src + static_cast<size_t>(l) * (2 * kHeadDim) + 4 * lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < kRopeF32Rows / 4; ++j) {
    const int rr = 4 * j + warp;
    tile[4 * lane + 0][rr] = x[j].x;
    tile[4 * lane + 1][rr] = x[j].y;
    tile[4 * lane + 2][rr] = x[j].z;
    tile[4 * lane + 3][rr] = x[j].w;
  }
  __syncthreads();
  // v^T row c = 4 i + warp: each lane writes key l0 + lane of it
  const int l = l0 + lane;
#pragma unroll 8
  for (int i = 0; i < (2 * kHeadDim) / 4; ++i) {
    const int c = 4 * i + warp;
    if (l < a.L_pad) dst[static_cast<size_t>(c) * a.L_pad + l] = l < a.L ? round_tf32(tile[c][lane]) : 0.0f;
  }
  __syncthreads();
}

// The FP32 pre-pass as a grid of resident blocks, each walking a contiguous chunk of items:
// first the RoPE items (positions [32 pb, 32 pb + 32) of one plane of q and of k; the thread of
// position row r and pair group g computes its 8 (cos, sin) once per position block), then the
// transpose items (32 keys of one v plane).
__global__ void __launch_bounds__(kRopeF32Threads, 8) rope_f32_kernel(RopeF32Args a) {
  // the attention grid may be scheduled now; it waits for this grid before reading its output
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float tile[2 * kHeadDim][kRopeF32Rows + 1];
  const long long n_pb = (a.L + kRopeF32Rows - 1) / kRopeF32Rows;
  const long long n_rope = a.q ? n_pb * a.planes : 0;
  const long long n_items = n_rope + (a.v ? n_pb * a.planes_v : 0);
  const long long per = (n_items + gridDim.x - 1) / gridDim.x;
  const long long i0 = static_cast<long long>(blockIdx.x) * per;
  const long long i1 = i0 + per < n_items ? i0 + per : n_items;
  const int r = threadIdx.x >> 2;
  const int g = threadIdx.x & 3;   // pairs [8g, 8g + 8)
  const size_t plane_stride = static_cast<size_t>(a.L) * kHeadDim;
  long long cur_pb = -1;
  float c[8], s[8];
  for (long long it = i0; it < i1; ++it) {
    if (it >= n_rope) {
      const long long j = it - n_rope;
      transpose_v_item(a, static_cast<int>(j / a.planes_v) * kRopeF32Rows, j % a.planes_v, tile);
      continue;
    }
    const long long pb = it / a.planes, pl = it % a.planes;
    const int l = static_cast<int>(pb) * kRopeF32Rows + r;
    if (l >= a.L) continue;
    const size_t off = static_cast<size_t>(pl) * plane_stride + static_cast<size_t>(l) * kHeadDim + 8 * g;
    // q and k of this row and pair group: all 8 loads before the first use
    float4 v4[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float* src = t == 0 ? a.q : a.k;
      v4[t][0] = ld_stream_f4(src + off);
      v4[t][1] = ld_stream_f4(src + off + 4);
      v4[t][2] = ld_stream_f4(src + off + 32);
      v4[t][3] = ld_stream_f4(src + off + 36);
    }
    if (pb != cur_pb) {
      cur_pb = pb;
      const int p = a.positions ? a.positions[l] : l;
      const float pf = static_cast<float>(p);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float theta = __fmul_rn(pf, a.inv_freq[8 * g + i]);
        sincosf(theta, &s[i], &c[i]);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float* dst = t == 0 ? a.q_out : a.k_out;
      float lo[8] = {v4[t][0].x, v4[t][0].y, v4[t][0].z, v4[t][0].w, v4[t][1].x, v4[t][1].y, v4[t][1].z, v4[t][1].w};
      float hi[8] = {v4[t][2].x, v4[t][2].y, v4[t][2].z, v4[t][2].w, v4[t][3].x, v4[t][3].y, v4[t][3].z, v4[t][3].w};
      rope_rotate8_f32(lo, hi, c, s);
      st_f4(dst + off, make_float4(lo[0], lo[1], lo[2], lo[3]));
      st_f4(dst + off + 4, make_float4(lo[4], lo[5], lo[6], lo[7]));
      st_f4(dst + off + 32, make_float4(hi[0], hi[1], hi[2], hi[3]));
      st_f4(dst + off + 36, make_float4(hi[4], hi[5], hi[6], hi[7]));
    }
  }
}

// ------------------------------------------------------------------------------ attention, TF32

constexpr int kBN = 64;                          // keys per tile
constexpr int kAtomQ = kBlockM * 128;            // one 128-row x 32-dim FP32 swizzle atom (16 KB)
constexpr int kAtomK = kBN * 128;                // one 64-row x 32-column FP32 atom (8 KB)
constexpr int kNS = 2;                           // K and V ring stages
constexpr int kQBytes = 4 * kAtomQ;              // Q: 2 maps x 2 atoms
constexpr int kKStage = 4 * kAtomK;              // K: 2 maps x 2 atoms
constexpr int kVStage = 2 * kAtomQ;              // v^T: 128 values x 64 keys, 2 atoms of 32 keys
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kNS * kKStage;
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2][2], p_full[2][2],
//           pv_done[2], o_full[2], drain[2]
constexpr int kNBar = 1 + 2 * kNS + 2 * kNS + 4 + 4 + 2 + 2 + 2;
constexpr int kOffBar = kOffV + kNS * kVStage;
constexpr int kOffMisc = kOffBar + 8 * kNBar;    // tmem base, abort flag
constexpr int kOffLsum = kOffMisc + 16;          // float [2][128]
constexpr int kSmemUsed = kOffLsum + 2 * kBlockM * 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 227 * 1024, "smem budget");
constexpr int kTmaWarp = 8, kMmaWarp = 9, kTmaWarpV = 11;

struct Bars {
  uint32_t q_full, k_full0, k_empty0, v_full0, v_empty0, s_full0, p_full0, pv_done0, o_full0, drain0;
  __device__ uint32_t k_full(int i) const { return k_full0 + 8 * i; }
  __device__ uint32_t k_empty(int i) const { return k_empty0 + 8 * i; }
  __device__ uint32_t v_full(int i) const { return v_full0 + 8 * i; }
  __device__ uint32_t v_empty(int i) const { return v_empty0 + 8 * i; }
  __device__ uint32_t s_full(int m, int b) const { return s_full0 + 8 * (2 * m + b); }
  __device__ uint32_t p_full(int m, int b) const { return p_full0 + 8 * (2 * m + b); }
  __device__ uint32_t pv_done(int m) const { return pv_done0 + 8 * m; }
  __device__ uint32_t o_full(int m) const { return o_full0 + 8 * m; }
  __device__ uint32_t drain(int m) const { return drain0 + 8 * m; }
};

__device__ __forceinline__ uint32_t s_col(int m, int b) { return 256 * m + 64 * b; }
__device__ __forceinline__ uint32_t o_col(int m) { return 256 * m + 128; }

// O_m *= f in tensor memory (the lazy rescale; rare, out of line).
__device__ __noinline__ void rescale_o128(uint32_t taddr, float f) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t o[32];
    tmem_ld32_nowait(taddr + 32 * cc, o);
    tmem_wait_ld_32(o);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float2 v2 = fmul2(make_float2(__uint_as_float(o[j]), __uint_as_float(o[j + 1])), make_float2(f, f));
      o[j] = __float_as_uint(v2.x);
      o[j + 1] = __float_as_uint(v2.y);
    }
    tmem_st32(taddr + 32 * cc, o);
  }
}

__global__ void __launch_bounds__(kFmhaThreads, 1)
    fmha_tf32_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FmhaF32Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + kOffQ, sK = sb + kOffK, sV = sb + kOffV;
  Bars bar;
  bar.q_full = sb + kOffBar;
  bar.k_full0 = bar.q_full + 8;
  bar.k_empty0 = bar.k_full0 + 8 * kNS;
  bar.v_full0 = bar.k_empty0 + 8 * kNS;
  bar.v_empty0 = bar.v_full0 + 8 * kNS;
  bar.s_full0 = bar.v_empty0 + 8 * kNS;
  bar.p_full0 = bar.s_full0 + 32;
  bar.pv_done0 = bar.p_full0 + 32;
  bar.o_full0 = bar.pv_done0 + 16;
  bar.drain0 = bar.o_full0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = a.L;
  const int unit = static_cast<int>(blockIdx.x);
  const int bh = unit / a.n_qblocks;
  const int q0 = (unit % a.n_qblocks) * kBlockM;
  const int q_last = min(L, q0 + kBlockM) - 1;
  const int w = a.window;
  // key tiles: all keys, or the block's window span [q0 - w, q_last + w] clipped to [0, L - 1]
  // and tiled from its first key
  int k_first = 0, t_hi = (L - 1) / kBN;
  if (w >= 0) {
    // rounded down to a multiple of 4 keys: a v^T tile copy then starts on a 16-byte boundary
    k_first = max(0, q0 - w) & ~3;
    t_hi = (min(L - 1, q_last + w) - k_first) / kBN;
  }
  const int n_tiles = t_hi + 1;
  const uint64_t tmo = a.timeout_ns;
  const uint64_t drain_tmo = tmo > 1000000000ull ? tmo : 1000000000ull;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full, 1);
    for (int i = 0; i < kNS; ++i) {
      mbar_init(bar.k_full(i), 1);
      mbar_init(bar.k_empty(i), 2);   // one commit from each MMA issuer
      mbar_init(bar.v_full(i), 1);
      mbar_init(bar.v_empty(i), 2);
    }
    for (int m = 0; m < 2; ++m) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar.s_full(m, b), 1);
        mbar_init(bar.p_full(m, b), 4);   // one elected arrival per softmax warp
      }
      mbar_init(bar.pv_done(m), 1);
      mbar_init(bar.o_full(m), 1);
      mbar_init(bar.drain(m), 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == kTmaWarpV && lane == 0) tma_prefetch_desc(&tm_v);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- Q and K producer
    // q', k' are the RoPE pass's output (programmatic dependent launch): wait for that grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    mbar_arrive_expect_tx_w(bar.q_full, kQBytes);
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int at = 0; at < 2; ++at)
        tma_load_3d_w(sQ + (2 * m + at) * kAtomQ, &tm_q, bar.q_full, 32 * at, q0, 2 * bh + m);
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int st = it % kNS;
      if (!pwait_w(bar.k_empty(st), ((it / kNS) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo)) break;
      const int key0 = k_first + it * kBN;
      const uint32_t dst = sK + st * kKStage;
      mbar_arrive_expect_tx_w(bar.k_full(st), kKStage);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int at = 0; at < 2; ++at)
          tma_load_3d_w(dst + (2 * m + at) * kAtomK, &tm_k, bar.k_full(st), 32 * at, key0, 2 * bh + m);
      issued = it + 1;
    }
    mbar_wait_limit(bar.q_full, 0, drain_tmo);
    for (int it = issued > kNS ? issued - kNS : 0; it < issued; ++it)
      mbar_wait_limit(bar.k_full(it % kNS), (it / kNS) & 1, drain_tmo);
    __syncwarp();
  } else if (warp == kTmaWarpV) {
    // ---------------------------------------------------------------- v^T producer
    // v^T is the pre-pass's output: wait for that grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int st = it % kNS;
      if (!pwait_w(bar.v_empty(st), ((it / kNS) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo)) break;
      const int key0 = k_first + it * kBN;
      const uint32_t dst = sV + st * kVStage;
      mbar_arrive_expect_tx_w(bar.v_full(st), kVStage);
#pragma unroll
      for (int at = 0; at < 2; ++at) tma_load_3d_w(dst + at * kAtomQ, &tm_v, bar.v_full(st), key0 + 32 * at, 0, bh);
      issued = it + 1;
    }
    for (int it = issued > kNS ? issued - kNS : 0; it < issued; ++it)
      mbar_wait_limit(bar.v_full(it % kNS), (it / kNS) & 1, drain_tmo);
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuer of map m
    const int m = warp - kMmaWarp;
    constexpr uint32_t idesc_s = make_idesc_tf32(kBlockM, kBN, false);
    constexpr uint32_t idesc_o = make_idesc_tf32(kBlockM, 2 * kHeadDim, false);
    // All operands K-major: an MMA reads 8 FP32 (32 bytes) of each row; a row's 64 values
    // (dims, or keys of v^T) are two 128-byte atoms, 16 KB apart for Q and v^T (128 rows), 8 KB
    // for K (64 rows).
    const uint64_t dq = smem_desc_sw128(sQ + 2 * m * kAtomQ, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sK + 2 * m * kAtomK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sV, 16, 1024);
    auto issue_s = [&](int it) {
      const int st = it % kNS;
      const uint64_t dk = dk0 + static_cast<uint64_t>(st * (kKStage >> 4));
      const uint32_t d = tmem + s_col(m, it & 1);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 8; ++kk)
        umma_ss_tf32_w(d, dq + (kk >> 2) * (kAtomQ >> 4) + 2 * (kk & 3), dk + (kk >> 2) * (kAtomK >> 4) + 2 * (kk & 3),
                       idesc_s, kk > 0 ? 1u : 0u);
      umma_commit_w(bar.s_full(m, it & 1));
      umma_commit_w(bar.k_empty(st));
    };
    const int eb = kErrMma;
    bool ok = pwait_w(bar.q_full, 0, abort_flag, a.err, eb, tmo) &&
              pwait_w(bar.k_full(0), 0, abort_flag, a.err, eb, tmo);
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
    if (ok && n_tiles > 1) {
      ok = pwait_w(bar.k_full(1 % kNS), (1 / kNS) & 1, abort_flag, a.err, eb, tmo);
      if (ok) {
        tc_fence_after();
        issue_s(1);
      }
    }
    for (int it = 0; ok && it < n_tiles; ++it) {
      const int sv = it % kNS;
      ok = pwait_w(bar.v_full(sv), (it / kNS) & 1, abort_flag, a.err, eb, tmo) &&
           pwait_w(bar.p_full(m, it & 1), (it >> 1) & 1, abort_flag, a.err, eb, tmo);
      if (!ok) break;
      tc_fence_after();
      const uint64_t dv = dv0 + static_cast<uint64_t>(sv * (kVStage >> 4));
      const uint32_t a_p = tmem + s_col(m, it & 1);
#pragma unroll
      for (int kk = 0; kk < kBN / 8; ++kk)
        umma_ts_tf32_w(tmem + o_col(m), a_p + 8 * kk, dv + (kk >> 2) * (kAtomQ >> 4) + 2 * (kk & 3), idesc_o,
                       (it > 0 || kk > 0) ? 1u : 0u);
      umma_commit_w(bar.pv_done(m));
      umma_commit_w(bar.v_empty(sv));
      if (it + 1 == n_tiles) umma_commit_w(bar.o_full(m));
      if (it + 2 < n_tiles) {
        // S(it + 2) goes into the buffer P(it) occupies: after P.V(it) has read it
        ok = pwait_w(bar.pv_done(m), it & 1, abort_flag, a.err, eb, tmo) &&
             pwait_w(bar.k_full((it + 2) % kNS), ((it + 2) / kNS) & 1, abort_flag, a.err, eb, tmo);
        if (!ok) break;
        tc_fence_after();
        issue_s(it + 2);
      }
    }
    umma_commit_w(bar.drain(m));
    mbar_wait_limit(bar.drain(m), 0, drain_tmo);
    __syncwarp();
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax of map m
    const int m = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int grow = q0 + r;
    const float c = a.scale_log2;
    const float tau = 8.0f / c;
    // this warp's 32 rows: a tile needs the element mask only if it is not wholly inside each of
    // their windows
    const int rows_lo = q0 + 32 * quarter, rows_hi = rows_lo + 31;
    float m_use = -INFINITY, l_sum = 0.0f;
    bool ok = true;
    for (int it = 0; it < n_tiles; ++it) {
      const int b = it & 1;
      ok = pwait(bar.s_full(m, b), (it >> 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = tmem + s_col(m, b) + lane_off;
      const int key0 = k_first + it * kBN;
      const bool need_mask = (key0 + kBN > L) || (w >= 0 && !(key0 >= rows_hi - w && key0 + kBN - 1 <= rows_lo + w));
      // this row's keys are columns [j_lo, j_hi) of the tile
      const int j_lo = w >= 0 ? grow - w - key0 : 0;
      const int j_hi = w >= 0 ? min(L - key0, grow + w + 1 - key0) : L - key0;
      if (need_mask && __all_sync(0xffffffffu, max(j_lo, 0) >= min(j_hi, kBN))) {
        // No row of this warp has a key in this tile: P = 0, and the rows' max and sum stay as
        // they are (exactly what the masked path gives); the warp goes on to its next tile.
        uint32_t z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0u;
        tmem_st32(sa, z);
        tmem_st32(sa + 32, z);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(m, b));
        continue;
      }
      uint32_t sr[kBN];
      float mt;
      tmem_ld64_max_nowait(sa, sr, mt);
      tmem_wait_ld_64_max(sr, mt);
      if (need_mask) {
        // The loaded maximum also covers the masked columns, so the row max is taken again over
        // the masked row.  The mask runs on the FMA pipe: a_j = sat(1 - j_lo + j) and
        // b_j = sat(j_hi - j) are both 1 exactly on the row's keys, and s_j + (a_j b_j - 1) 2^100
        // leaves those scores exact and puts every other one far below any score (its
        // exponential is 0, as for -inf); a row with no key here gets -inf as its max.
        const float fa = static_cast<float>(1 - j_lo), fb = static_cast<float>(j_hi);
#pragma unroll
        for (int j = 0; j < kBN; j += 2) {
          const float2 a2 = make_float2(sat_add(fa, static_cast<float>(j)), sat_add(fa, static_cast<float>(j + 1)));
          const float2 b2 = make_float2(sat_add(fb, -static_cast<float>(j)), sat_add(fb, -static_cast<float>(j + 1)));
          const float2 w2 = ffma2(a2, b2, make_float2(-1.0f, -1.0f));
          const float2 s2 = ffma2(w2, make_float2(0x1p100f, 0x1p100f),
                                  make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])));
          sr[j] = __float_as_uint(s2.x);
          sr[j + 1] = __float_as_uint(s2.y);
        }
        // 8 independent chains; chain q covers elements q, q + 8, ..., q + 56
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(__uint_as_float(sr[q]), __uint_as_float(sr[q + 8]));
#pragma unroll
        for (int j = 16; j < kBN; j += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], __uint_as_float(sr[j + q]), __uint_as_float(sr[j + 8 + q]));
        }
        mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        if (mt < -0x1p99f) mt = -INFINITY;
      }
      float f = 1.0f;
      bool rescale = false;
      if (it == 0) {
        m_use = mt;
      } else if (__any_sync(0xffffffffu, mt > m_use + tau)) {
        const float m_new = fmaxf(m_use, mt);
        // a row whose running max is still -inf has had P = 0 on every tile so far: its O row
        // and row sum are exactly 0 and need no rescale (nor the wait for the last P.V)
        f = (m_new == m_use || m_use == -INFINITY) ? 1.0f : ex2_approx((m_use - m_new) * c);
        m_use = m_new;
        rescale = __any_sync(0xffffffffu, f != 1.0f);
      }
      const float mb = (m_use == -INFINITY) ? 0.0f : m_use * c;
      const float2 c2 = make_float2(c, c), nmb2 = make_float2(-mb, -mb);
      float2 sum0 = make_float2(0.0f, 0.0f), sum1 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int e = 0; e < kBN; e += 4) {
        const float2 x0 = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nmb2);
        const float2 x1 = ffma2(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2, nmb2);
        const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
        const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
        sum0 = fadd2(sum0, p0);
        sum1 = fadd2(sum1, p1);
        sr[e] = __float_as_uint(round_tf32(p0.x));
        sr[e + 1] = __float_as_uint(round_tf32(p0.y));
        sr[e + 2] = __float_as_uint(round_tf32(p1.x));
        sr[e + 3] = __float_as_uint(round_tf32(p1.y));
      }
      const float2 sum = fadd2(sum0, sum1);
      l_sum = fmaf(l_sum, f, sum.x + sum.y);
      if (rescale) {
        // O_m is still written by P.V of the previous tile until it is done
        ok = pwait(bar.pv_done(m), (it - 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        rescale_o128(tmem + o_col(m) + lane_off, f);
      }
      // P over S in this buffer (the A operand of P.V)
      tmem_st32(sa, sr);
      tmem_st32(sa + 32, sr + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_full(m, b));
    }

    // ---------------------------------------------------------------- epilogue
    if (ok) ok = pwait(bar.o_full(0), 0, abort_flag, a.err, kErrSoftmax, tmo);
    if (ok) ok = pwait(bar.o_full(1), 0, abort_flag, a.err, kErrSoftmax, tmo);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    lsum[m * kBlockM + r] = l_sum;
    tc_fence_before();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    tc_fence_after();
    const float l0 = lsum[r], l1 = lsum[kBlockM + r];
    const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f;
    const float inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
    const float lam = a.lambda[bh % a.H];
    float* dst = a.out + (static_cast<size_t>(bh) * L + grow) * static_cast<size_t>(2 * kHeadDim) + 64 * m;
    if (ok) {
      // warpgroup m writes output columns [64 m, 64 m + 64)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t col = 64 * m + 32 * cc;
        uint32_t o0[32], o1[32];
        tmem_ld32_nowait(tmem + o_col(0) + lane_off + col, o0);
        tmem_ld32_nowait(tmem + o_col(1) + lane_off + col, o1);
        tmem_wait_ld_32(o0);
        tmem_wait_ld_32(o1);
        if (grow < L) {
          float4* d4 = reinterpret_cast<float4*>(dst + 32 * cc);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float y[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
              y[t] = fmaf(-lam, __uint_as_float(o1[4 * j + t]) * inv1, __uint_as_float(o0[4 * j + t]) * inv0);
            d4[j] = make_float4(y[0], y[1], y[2], y[3]);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t rope_f32_launch(const RopeF32Args& a, int num_sms, cudaStream_t stream) {
  // one block per resident slot (the occupancy calculator's count, looked up once)
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rope_f32_kernel, kRopeF32Threads, 0) != cudaSuccess || n < 1)
      n = 1;
    return n;
  }();
  const long long n_pb = (a.L + kRopeF32Rows - 1) / kRopeF32Rows;
  const long long items = n_pb * ((a.q ? a.planes : 0) + (a.v ? a.planes_v : 0));
  long long grid = static_cast<long long>(per_sm) * num_sms;
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  rope_f32_kernel<<<static_cast<unsigned>(grid), kRopeF32Threads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t fmha_tf32_set_attributes() {
  return cudaFuncSetAttribute(fmha_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
}

bool fmha_tf32_check(int* regs) {
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, fmha_tf32_kernel) != cudaSuccess) return false;
  *regs = attr.numRegs;
  return attr.binaryVersion == 103;
}

cudaError_t fmha_tf32_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FmhaF32Args& a, long long num_ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
  cfg.blockDim = dim3(kFmhaThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fmha_tf32_kernel, tq, tk, tv, a);
}

}  // namespace sa
