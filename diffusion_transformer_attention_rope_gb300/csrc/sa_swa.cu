// sa_swa.cu -- differential attention with a narrow symmetric sliding window for sm_103a
// (GB300): SAME-L's diff_attn_swa at its own window of +-17 (HF discussion #6 "sm_120 SAME-L",
// "Three gotchas": a key tile much wider than the window is mostly masked-out waste, and the
// kernel there is faster with small tiles).  Same result as the general attention kernel:
//   out = softmax(q1' k1'^T / sqrt(d)) v - lambda_h * softmax(q2' k2'^T / sqrt(d)) v
// over the keys |i - j| <= w, RoPE of q in the prologue (FP32, cast back; after the QK-RMSNorm
// when one is asked for), softmax in FP32, the subtraction in FP32 on the FP32 accumulators.
//
// With a narrow window a query block touches only a few key tiles, so the general kernel's
// fixed costs per CTA (setup, Q load and rotation, pipeline fill, drain, epilogue, relaunch)
// outweigh its key loop.  Here one CTA per SM walks a contiguous run of query blocks (units):
//   - 64-key tiles (the span of a 128-row block at +-17 is 162 keys: 3 tiles of 64 instead of 2
//     of 128), S double-buffered per map in tensor memory and P (fp16/bf16) written over its S
//     buffer, the A operand of a TS P.V MMA, so P never goes through shared memory;
//   - Q double-buffered in shared memory: the next unit's raw Q arrives while this one runs
//     (the first two units' Q are copied before the wait for the K pass; the V ring starts
//     once the first Q has landed);
//   - the rings, S buffers and their barriers run on across units with a CTA-wide tile count
//     (the P.V completion is tracked per S buffer, so an S MMA waits only for the P.V that read
//     its buffer), and the issuers run the S MMAs two tiles ahead of the P.V MMAs across unit
//     boundaries; the first P.V of a unit (which overwrites O) waits until the previous
//     epilogue has read O;
//   - the RoPE of each unit's Q and each unit's epilogue run on a warpgroup of their own (the
//     output warps), so the softmax warps go from one unit's last key tile straight to the next
//     unit's first: the output warps rotate unit u + 1's Q while the softmax warps work on unit
//     u, and write unit u's output while they work on unit u + 1.
// Warp roles (512 threads): warps 0-3 / 4-7 softmax of map 0 / 1 (thread = query row = TMEM
// lane), warp 8 TMA of Q and the K ring, warp 9 TMEM allocation and MMA issuer of map 0, warp 10
// MMA issuer of map 1, warp 11 TMA of the V ring, warps 12-15 the output warps (thread = query
// row of both maps).
// Tensor memory (512 columns): map m at 256 m: S buffer 0 | S buffer 1 | O = 64 | 64 | 128.
// Shared memory: Q 2 x 32 KB, K ring 3 x 16 KB, V ring 3 x 16 KB, output staging 32 KB (each
// output warp writes its 32 rows x 128 values with two TMA stores, not as scattered 16-byte
// stores of rows 256 bytes apart).  Every wait is bounded.
#include <cuda.h>

#include "sa_kernels.h"
#include "sa_pipe.cuh"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kSwaThreads = 512;               // 4 warpgroups: 2 softmax, control, output
constexpr int kOutWarp = 12;                   // first output warp
constexpr int kBN = 64;                        // keys per tile
constexpr int kQTile = kBlockM * kHeadDim * 2; // one map's 128 x 64 Q tile (16 KB, one atom)
constexpr int kKMap = kBN * kHeadDim * 2;      // one map's 64 x 64 K tile (8 KB)
constexpr int kNS = 3;                         // K and V ring stages
constexpr int kQBuf = 2 * kQTile;              // both maps
constexpr int kKStage = 2 * kKMap;             // both maps
constexpr int kVStage = kBN * 2 * kHeadDim * 2;// 64 keys x 128 values (two 8 KB atoms)
constexpr int kVAtom = kVStage / 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kQBuf;
constexpr int kOffV = kOffK + kNS * kKStage;
// output staging for the epilogue's TMA stores: per output warp 32 rows x 128 values as two
// 32 x 64 boxes of 4 KB
constexpr int kStageBox = 32 * 128;
constexpr int kStageWarp = 2 * kStageBox;
constexpr int kOffStage = kOffV + kNS * kVStage;
// barriers: q_full[2], q_ready[2][2], q_free[2], k_full[kNS], k_empty[kNS], v_full[kNS],
//           v_empty[kNS], s_full[2][2], p_full[2][2], pv_done[2][2], o_full[2], o_free, drain[2],
//           l_ready[2], l_free[2]
constexpr int kNBar = 2 + 4 + 2 + 4 * kNS + 4 + 4 + 4 + 2 + 1 + 2 + 2 + 2;
constexpr int kOffBar = kOffStage + 4 * kStageWarp;
constexpr int kOffMisc = kOffBar + 8 * kNBar;  // tmem base, abort flag
constexpr int kOffLsum = kOffMisc + 16;        // float [2 units][2 maps][128]
constexpr int kSmemUsed = kOffLsum + 2 * 2 * kBlockM * 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 227 * 1024, "smem budget");
constexpr int kTmaWarp = 8, kMmaWarp = 9, kTmaWarpV = 11;

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full(int b) const { return base + 8 * b; }
  __device__ uint32_t q_ready(int b, int m) const { return base + 16 + 8 * (2 * b + m); }
  __device__ uint32_t q_free(int b) const { return base + 48 + 8 * b; }
  __device__ uint32_t k_full(int i) const { return base + 64 + 8 * i; }
  __device__ uint32_t k_empty(int i) const { return base + 64 + 8 * kNS + 8 * i; }
  __device__ uint32_t v_full(int i) const { return base + 64 + 16 * kNS + 8 * i; }
  __device__ uint32_t v_empty(int i) const { return base + 64 + 24 * kNS + 8 * i; }
  __device__ uint32_t s_full(int m, int b) const { return base + 64 + 32 * kNS + 8 * (2 * m + b); }
  __device__ uint32_t p_full(int m, int b) const { return base + 96 + 32 * kNS + 8 * (2 * m + b); }
  // P.V completion of map m, per S buffer b (the P.V of tile g commits pv_done(m, g & 1))
  __device__ uint32_t pv_done(int m, int b) const { return base + 128 + 32 * kNS + 8 * (2 * m + b); }
  __device__ uint32_t o_full(int m) const { return base + 160 + 32 * kNS + 8 * m; }
  __device__ uint32_t o_free() const { return base + 176 + 32 * kNS; }
  __device__ uint32_t drain(int m) const { return base + 184 + 32 * kNS + 8 * m; }
  // the row sums of the units of parity b: written by the softmax warps (l_ready), read by the
  // output warps (l_free)
  __device__ uint32_t l_ready(int b) const { return base + 200 + 32 * kNS + 8 * b; }
  __device__ uint32_t l_free(int b) const { return base + 216 + 32 * kNS + 8 * b; }
};
static_assert(232 + 32 * kNS == 8 * kNBar, "barrier layout");

__device__ __forceinline__ uint32_t s_col(int m, int b) { return 256 * m + 64 * b; }
__device__ __forceinline__ uint32_t o_col(int m) { return 256 * m + 128; }

// A unit (128 query rows of one (batch, head), both maps) and the key tiles it visits: the
// window span [q0 - w, q_last + w] clipped to [0, L - 1], tiled from its first key.
struct Unit {
  int bh, q0, k_first, n_tiles;
};

__device__ __forceinline__ Unit unit_at(const FmhaSwaArgs& a, int bh, int q0) {
  Unit x;
  x.bh = bh;
  x.q0 = q0;
  const int q_last = min(a.L, q0 + kBlockM) - 1;
  x.k_first = max(0, q0 - a.window);
  x.n_tiles = (min(a.L - 1, q_last + a.window) - x.k_first) / kBN + 1;
  return x;
}

// Unit u (one 64-bit division, at the start of a run only).
__device__ __forceinline__ Unit unit_of(const FmhaSwaArgs& a, long long u) {
  return unit_at(a, static_cast<int>(u / a.n_qblocks), static_cast<int>(u % a.n_qblocks) * kBlockM);
}

// The unit after x in the run (the next query block, or the next (batch, head)'s first).
__device__ __forceinline__ Unit next_unit(const FmhaSwaArgs& a, const Unit& x) {
  return x.q0 + kBlockM < a.L ? unit_at(a, x.bh, x.q0 + kBlockM) : unit_at(a, x.bh + 1, 0);
}

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

// RoPE of this thread's raw Q rows of both maps in shared memory (128-byte-swizzled; the rows
// share the position), with the (cos, sin) table of the RoPE pass and its arithmetic
// (rope_rotate8), so that q' has the pass's bits; with NORM each row is QK-RMS-normalised first,
// with the pass's sum order and scaling.  Each table entry is loaded once for both rows: all 16
// up front, or (NORM, which needs the registers for its scales) one group of 4 at a time.
template <bool BF16, bool NORM>
__device__ __noinline__ void rotate_q_rows(const float2* cs, int cs_stride, int L, int grow, uint32_t row0,
                                           uint32_t row1, int r, const float* gamma, float eps) {
  if (grow >= L) return;
  const float4* cs4 = reinterpret_cast<const float4*>(cs) + grow;
  auto rotate_group = [&](uint32_t row, int g, const float4 (&t)[4], float inv) {
    const uint4 lo = ld_shared_v4(row + ((g ^ (r & 7)) << 4));
    const uint4 hi = ld_shared_v4(row + (((g + 4) ^ (r & 7)) << 4));
    float cg[8], sg[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cg[2 * i] = t[i].x;
      cg[2 * i + 1] = t[i].y;
      sg[2 * i] = t[i].z;
      sg[2 * i + 1] = t[i].w;
    }
    uint4 olo, ohi;
    if (NORM) {
      float sl[8], sh[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sl[i] = __fmul_rn(inv, gamma[8 * g + i]);
        sh[i] = __fmul_rn(inv, gamma[32 + 8 * g + i]);
      }
      rope_rotate8_scaled<BF16>(lo, hi, cg, sg, sl, sh, olo, ohi);
    } else {
      rope_rotate8<BF16>(lo, hi, cg, sg, olo, ohi);
    }
    st_shared_v4(row + ((g ^ (r & 7)) << 4), olo.x, olo.y, olo.z, olo.w);
    st_shared_v4(row + (((g + 4) ^ (r & 7)) << 4), ohi.x, ohi.y, ohi.z, ohi.w);
  };
  if (NORM) {
    // each row's 1 / rms from its raw values, then the rotation group by group
    float inv[2];
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      const uint32_t row = mm ? row1 : row0;
      float tg[4];
#pragma unroll
      for (int g = 0; g < 4; ++g)
        tg[g] = sumsq8<BF16>(ld_shared_v4(row + ((g ^ (r & 7)) << 4))) +
                sumsq8<BF16>(ld_shared_v4(row + (((g + 4) ^ (r & 7)) << 4)));
      inv[mm] = qknorm_inv_rms((tg[0] + tg[1]) + (tg[2] + tg[3]), eps);
    }
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      float4 t[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) t[i] = __ldg(cs4 + static_cast<size_t>(4 * g + i) * cs_stride);
      rotate_group(row0, g, t, inv[0]);
      rotate_group(row1, g, t, inv[1]);
    }
  } else {
    float4 t[4][4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i) t[g][i] = __ldg(cs4 + static_cast<size_t>(4 * g + i) * cs_stride);
#pragma unroll 1
    for (int mm = 0; mm < 2; ++mm) {
#pragma unroll
      for (int g = 0; g < 4; ++g) rotate_group(mm ? row1 : row0, g, t[g], 1.0f);
    }
  }
}

// NORM: the QK-RMSNorm form (a kernel of its own, so that the plain one carries none of its code)
template <bool BF16, bool NORM>
__global__ void __launch_bounds__(kSwaThreads, 1)
    fmha_swa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ FmhaSwaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + kOffQ, sK = sb + kOffK, sV = sb + kOffV;
  Bars bar;
  bar.base = sb + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = a.L;
  // this CTA's run of units
  const long long u_begin = static_cast<long long>(blockIdx.x) * a.units / gridDim.x;
  const long long u_end = static_cast<long long>(blockIdx.x + 1) * a.units / gridDim.x;
  const int n_units = static_cast<int>(u_end - u_begin);
  const uint64_t tmo = a.timeout_ns;
  const uint64_t drain_tmo = tmo > 1000000000ull ? tmo : 1000000000ull;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.q_full(b), 1);
      mbar_init(bar.q_ready(b, 0), 4);   // one elected arrival per softmax warp of the map
      mbar_init(bar.q_ready(b, 1), 4);
      mbar_init(bar.q_free(b), 2);       // one commit from each MMA issuer
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(bar.k_full(i), 1);
      mbar_init(bar.k_empty(i), 2);
      mbar_init(bar.v_full(i), 1);
      mbar_init(bar.v_empty(i), 2);
    }
    for (int m = 0; m < 2; ++m) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar.s_full(m, b), 1);
        mbar_init(bar.p_full(m, b), 4);
      }
      mbar_init(bar.pv_done(m, 0), 1);
      mbar_init(bar.pv_done(m, 1), 1);
      mbar_init(bar.o_full(m), 1);
      mbar_init(bar.drain(m), 1);
    }
    mbar_init(bar.o_free(), 4);          // every output warp, after the epilogue read O
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar.l_ready(b), 8);      // every softmax warp, after writing its row sums
      mbar_init(bar.l_free(b), 4);       // every output warp, after reading them
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
  if (warp == kOutWarp && lane == 0) tma_prefetch_desc(&tm_o);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- Q and K producer
    int g = 0, issued = 0, q_issued = 0;
    bool ok = true;
    Unit x = unit_of(a, u_begin);
    auto load_q = [&](int ui, const Unit& y) {
      const int qb = ui & 1;
      mbar_arrive_expect_tx_w(bar.q_full(qb), kQBuf);
      tma_load_3d_w(sQ + qb * kQBuf, &tm_q, bar.q_full(qb), 0, y.q0, 2 * y.bh);
      tma_load_3d_w(sQ + qb * kQBuf + kQTile, &tm_q, bar.q_full(qb), 0, y.q0, 2 * y.bh + 1);
      q_issued = ui + 1;
    };
    // Raw q is the caller's: the first two units' Q are copied before the wait for the RoPE
    // pass, whose output (k', or q' as well when cs is nullptr) the rest waits for
    // (programmatic dependent launch).
    if (a.cs != nullptr && n_units > 0) {
      load_q(0, x);
      if (n_units > 1) load_q(1, next_unit(a, x));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int ui = 0; ok && ui < n_units; ++ui, x = next_unit(a, x)) {
      const int qb = ui & 1;
      // the buffer's previous unit (ui - 2) must be done with it (its S MMAs have completed)
      if (ui >= q_issued) {
        if (ui >= 2 && !pwait_w(bar.q_free(qb), ((ui >> 1) - 1) & 1, abort_flag, a.err, kErrProducer, tmo)) break;
        load_q(ui, x);
      }
      for (int t = 0; t < x.n_tiles; ++t, ++g) {
        const int st = g % kNS;
        if (!pwait_w(bar.k_empty(st), ((g / kNS) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo)) {
          ok = false;
          break;
        }
        const int key0 = x.k_first + t * kBN;
        const uint32_t dst = sK + st * kKStage;
        mbar_arrive_expect_tx_w(bar.k_full(st), kKStage);
        tma_load_3d_w(dst, &tm_k, bar.k_full(st), 0, key0, 2 * x.bh);
        tma_load_3d_w(dst + kKMap, &tm_k, bar.k_full(st), 0, key0, 2 * x.bh + 1);
        issued = g + 1;
      }
    }
    // copies still in flight land before the CTA's shared memory goes away
    for (int i = issued > kNS ? issued - kNS : 0; i < issued; ++i)
      mbar_wait_limit(bar.k_full(i % kNS), (i / kNS) & 1, drain_tmo);
    for (int ui = q_issued > 2 ? q_issued - 2 : 0; ui < q_issued; ++ui)
      mbar_wait_limit(bar.q_full(ui & 1), (ui >> 1) & 1, drain_tmo);
    __syncwarp();
  } else if (warp == kTmaWarpV) {
    // ---------------------------------------------------------------- V producer
    int g = 0, issued = 0;
    // V is first read by the first P.V, well after the first Q: its copies start once that Q
    // has landed, so that the Q copies at the start of the kernel do not share HBM with them
    bool ok = n_units == 0 || pwait_w(bar.q_full(0), 0, abort_flag, a.err, kErrProducer, tmo);
    Unit x = unit_of(a, u_begin);
    for (int ui = 0; ok && ui < n_units; ++ui, x = next_unit(a, x)) {
      for (int t = 0; t < x.n_tiles; ++t, ++g) {
        const int st = g % kNS;
        if (!pwait_w(bar.v_empty(st), ((g / kNS) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo)) {
          ok = false;
          break;
        }
        const int key0 = x.k_first + t * kBN;
        const uint32_t dst = sV + st * kVStage;
        mbar_arrive_expect_tx_w(bar.v_full(st), kVStage);
        tma_load_3d_w(dst, &tm_v, bar.v_full(st), 0, key0, x.bh);
        tma_load_3d_w(dst + kVAtom, &tm_v, bar.v_full(st), 64, key0, x.bh);
        issued = g + 1;
      }
    }
    for (int i = issued > kNS ? issued - kNS : 0; i < issued; ++i)
      mbar_wait_limit(bar.v_full(i % kNS), (i / kNS) & 1, drain_tmo);
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuer of map m
    const int m = warp - kMmaWarp;
    constexpr uint32_t idesc_s = make_idesc_f16(kBlockM, kBN, BF16, false);
    constexpr uint32_t idesc_o = make_idesc_f16(kBlockM, 2 * kHeadDim, BF16, true);
    // K-major Q and K (one 128-byte atom per row: an MMA of K = 16 reads 32 bytes of it); V
    // MN-major, its 128 values two atoms 8 KB apart, 8-key groups 1 KB apart.
    const uint64_t dq0 = smem_desc_sw128(sQ + m * kQTile, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sK + m * kKMap, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sV, kVAtom, 1024);
    const int eb = kErrMma;
    auto issue_s = [&](int gg, uint64_t dq) {
      const int st = gg % kNS;
      const uint64_t dk = dk0 + static_cast<uint64_t>(st * (kKStage >> 4));
      const uint32_t d = tmem + s_col(m, gg & 1);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk) umma_ss_w(d, dq + 2 * kk, dk + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
      umma_commit_w(bar.s_full(m, gg & 1));
      umma_commit_w(bar.k_empty(st));
    };
    // S MMAs run ahead of the P.V MMAs by two tiles across unit boundaries: S(j) is issued as soon
    // as its buffer (that of tile j - 2) has been read by P.V(j - 2), whichever unit tile j belongs
    // to, so the softmax warps find the next unit's first S ready when they finish a unit.
    Unit sx = unit_of(a, u_begin);   // unit of the next S to issue
    int s_ui = 0, s_t = 0, s_g = 0;  // its index in the run, its tile in the unit, its tile in the run
    auto issue_next_s = [&]() {
      if (s_ui >= n_units) return true;
      const int qb = s_ui & 1;
      // a unit's first S: its Q has been rotated
      if (s_t == 0 && !pwait_w(bar.q_ready(qb, m), (s_ui >> 1) & 1, abort_flag, a.err, eb, tmo)) return false;
      // S(j) goes into the buffer of tile j - 2: after that tile's P.V has read its P
      if (s_g >= 2 && !pwait_w(bar.pv_done(m, s_g & 1), ((s_g - 2) >> 1) & 1, abort_flag, a.err, eb, tmo))
        return false;
      if (!pwait_w(bar.k_full(s_g % kNS), (s_g / kNS) & 1, abort_flag, a.err, eb, tmo)) return false;
      tc_fence_after();
      issue_s(s_g, dq0 + static_cast<uint64_t>(qb * (kQBuf >> 4)));
      // the unit's last S MMA is the last reader of its Q buffer: the next Q may land there once
      // it has completed
      if (s_t + 1 == sx.n_tiles) umma_commit_w(bar.q_free(qb));
      ++s_g;
      if (++s_t == sx.n_tiles) {
        s_t = 0;
        ++s_ui;
        sx = next_unit(a, sx);
      }
      return true;
    };
    bool ok = issue_next_s() && issue_next_s();
    int g = 0;
    Unit x = unit_of(a, u_begin);
    for (int ui = 0; ok && ui < n_units; ++ui, x = next_unit(a, x)) {
      const int n = x.n_tiles;
      for (int t = 0; t < n; ++t) {
        const int gg = g + t;
        const int sv = gg % kNS;
        ok = pwait_w(bar.v_full(sv), (gg / kNS) & 1, abort_flag, a.err, eb, tmo) &&
             pwait_w(bar.p_full(m, gg & 1), (gg >> 1) & 1, abort_flag, a.err, eb, tmo);
        // the first P.V of a unit overwrites O: the previous unit's epilogue must have read it
        if (ok && t == 0 && ui > 0) ok = pwait_w(bar.o_free(), (ui - 1) & 1, abort_flag, a.err, eb, tmo);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(sv * (kVStage >> 4));
        const uint32_t a_p = tmem + s_col(m, gg & 1);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts_w(tmem + o_col(m), a_p + 8 * kk, dv + 128 * kk, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(bar.pv_done(m, gg & 1));
        umma_commit_w(bar.v_empty(sv));
        if (t + 1 == n) umma_commit_w(bar.o_full(m));
        // S(gg + 2), of this unit or of the next ones
        ok = issue_next_s();
        if (!ok) break;
      }
      g += n;
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
    const float c = a.scale_log2;
    const float tau = 8.0f / c;
    const int w = a.window;
    int g = 0;
    bool ok = true;
    Unit x = unit_of(a, u_begin);
    for (int ui = 0; ok && ui < n_units; ++ui, x = next_unit(a, x)) {
      const int grow = x.q0 + r;
      // this warp's 32 rows: a tile needs the element mask only if it is not wholly inside each
      // of their windows
      const int rows_lo = x.q0 + 32 * quarter, rows_hi = rows_lo + 31;

      float m_use = -INFINITY, l_sum = 0.0f;
      for (int t = 0; t < x.n_tiles; ++t) {
        const int gg = g + t;
        const int b = gg & 1;
        ok = pwait(bar.s_full(m, b), (gg >> 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = tmem + s_col(m, b) + lane_off;
        const int key0 = x.k_first + t * kBN;
        const bool need_mask = (key0 + kBN > L) || !(key0 >= rows_hi - w && key0 + kBN - 1 <= rows_lo + w);
        // this row's keys are columns [j_lo, j_hi) of the tile
        const int j_lo = grow - w - key0;
        const int j_hi = min(L - key0, grow + w + 1 - key0);
        if (need_mask && __all_sync(0xffffffffu, max(j_lo, 0) >= min(j_hi, kBN))) {
          // No row of this warp has a key in this tile (the band of 32 rows misses it): P = 0,
          // and the rows' max and sum stay as they are (exactly what the masked path gives).
          // The warp goes straight on to its next tile, so on a narrow band the warps whose
          // rows miss a unit's first or last tile run ahead of the others.
          uint32_t z[kBN / 2];
#pragma unroll
          for (int j = 0; j < kBN / 2; ++j) z[j] = 0u;
          tmem_st32(sa, z);
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
          // The loaded maximum also covers the masked columns, so the row max is taken again
          // over the masked row.  The mask runs on the FMA pipe (the ALU pipe, half as wide, is
          // the one the compares and selects would load): a_j = sat(1 - j_lo + j) and
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
        if (t == 0) {
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
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int j = 0; j < kBN / 2; j += 2) {
          const int e = 2 * j;
          const float2 x0 = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nmb2);
          const float2 x1 = ffma2(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2, nmb2);
          const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
          const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
          sum0 = fadd2(sum0, p0);
          sum1 = fadd2(sum1, p1);
          pk[j] = pack2<BF16>(p0.x, p0.y);
          pk[j + 1] = pack2<BF16>(p1.x, p1.y);
        }
        const float2 sum = fadd2(sum0, sum1);
        l_sum = fmaf(l_sum, f, sum.x + sum.y);
        if (rescale) {
          // O_m is still written by P.V of the previous tile until it is done
          ok = pwait(bar.pv_done(m, (gg - 1) & 1), ((gg - 1) >> 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          rescale_o128(tmem + o_col(m) + lane_off, f);
        }
        // P over S in this buffer (the A operand of P.V)
        tmem_st32(sa, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(m, b));
      }
      if (!ok) break;
      // the unit's row sums go to the output warps (the buffer of this parity is free once they
      // have read the sums of unit ui - 2)
      if (ui >= 2) {
        ok = pwait(bar.l_free(ui & 1), ((ui >> 1) - 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      lsum[(ui & 1) * 2 * kBlockM + m * kBlockM + r] = l_sum;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.l_ready(ui & 1));
      g += x.n_tiles;
    }
  } else if (warp >= kOutWarp) {
    // ---------------------------------------------------------------- output warps
    // Thread = query row r of both maps.  Per unit: the RoPE of the next unit's Q (both maps),
    // then this unit's epilogue, out = O_0 / l_0 - lambda_h O_1 / l_1 in FP32, one RNE cast.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t stage = sb + kOffStage + (warp - kOutWarp) * kStageWarp;
    // a per-call (cos, sin) table is the RoPE pass's output
    if (!a.cs_static) asm volatile("griddepcontrol.wait;" ::: "memory");
    // RoPE of row r of unit ui's Q (both maps, in its buffer), then the Q goes to the issuers
    auto q_prologue = [&](int ui, const Unit& y) {
      const int qb = ui & 1;
      if (a.cs != nullptr && y.q0 + r < L) {
        // the row's 16 table entries into L2 while the Q copy is in flight
        const float4* cs4 = reinterpret_cast<const float4*>(a.cs) + y.q0 + r;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(cs4 + static_cast<size_t>(i) * a.cs_stride));
      }
      bool good = pwait(bar.q_full(qb), (ui >> 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
      good = __all_sync(0xffffffffu, good);
      if (!good) return false;
      if (a.cs != nullptr)
        rotate_q_rows<BF16, NORM>(a.cs, a.cs_stride, L, y.q0 + r, sQ + qb * kQBuf + r * 128,
                                  sQ + qb * kQBuf + kQTile + r * 128, r, a.gamma_q, a.eps);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar.q_ready(qb, 0));
        mbar_arrive(bar.q_ready(qb, 1));
      }
      return true;
    };
    Unit x = unit_of(a, u_begin);
    bool ok = n_units > 0 ? q_prologue(0, x) : true;
    for (int ui = 0; ok && ui < n_units; ++ui, x = next_unit(a, x)) {
      // lambda_h now: its load latency then stays off the path from O ready to O released
      const float lam = a.lambda[x.bh % a.H];
      // the next unit's Q first: its S MMAs then start as soon as this unit's last tiles free
      // the S buffers
      if (ui + 1 < n_units && !q_prologue(ui + 1, next_unit(a, x))) {
        ok = false;
        break;
      }
      // ---------------------------------------------------------------- epilogue of unit ui
      ok = pwait(bar.l_ready(ui & 1), (ui >> 1) & 1, abort_flag, a.err, kErrSoftmax, tmo);
      if (ok) ok = pwait(bar.o_full(0), ui & 1, abort_flag, a.err, kErrSoftmax, tmo);
      if (ok) ok = pwait(bar.o_full(1), ui & 1, abort_flag, a.err, kErrSoftmax, tmo);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* ls = lsum + (ui & 1) * 2 * kBlockM;
      const float l0 = ls[r], l1 = ls[kBlockM + r];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.l_free(ui & 1));
      const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f;
      const float inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
      // out = O_0 inv0 + O_1 (-lambda_h inv1), two elements per paired FP32 multiply and fma
      const float2 a2 = make_float2(inv0, inv0);
      const float nb = -lam * inv1;
      const float2 b2 = make_float2(nb, nb);
      // this warp's 32 rows x 128 values go through its staging block (two 32 x 64 boxes,
      // 128-byte swizzle: 16-byte chunk c of row i at c ^ (i & 7)) and two TMA stores
      if (lane == 0) bulk_wait_read();   // the previous unit's stores have read the block
      __syncwarp();
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o0[32], o1[32];
        tmem_ld32_nowait(tmem + o_col(0) + lane_off + 32 * cc, o0);
        tmem_ld32_nowait(tmem + o_col(1) + lane_off + 32 * cc, o1);
        tmem_wait_ld_32(o0);
        tmem_wait_ld_32(o1);
        if (cc == 3) {
          // O has been read: the next unit's first P.V may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar.o_free());
        }
        uint32_t pkd[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 y = ffma2(make_float2(__uint_as_float(o1[2 * j]), __uint_as_float(o1[2 * j + 1])), b2,
                                 fmul2(make_float2(__uint_as_float(o0[2 * j]), __uint_as_float(o0[2 * j + 1])), a2));
          pkd[j] = pack2<BF16>(y.x, y.y);
        }
        const uint32_t row = stage + (cc >> 1) * kStageBox + lane * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(row + (((4 * (cc & 1) + j) ^ (lane & 7)) << 4), pkd[4 * j], pkd[4 * j + 1], pkd[4 * j + 2],
                       pkd[4 * j + 3]);
      }
      // the staging block is complete: the TMA stores may read it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        // rows past L are outside the tensor and not written
        tma_store_3d(&tm_o, stage, 0, x.q0 + 32 * quarter, x.bh);
        tma_store_3d(&tm_o, stage + kStageBox, 64, x.q0 + 32 * quarter, x.bh);
        bulk_commit();
      }
    }
    // the output stores complete before the CTA's shared memory goes away
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16, bool NORM>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                   const FmhaSwaArgs& a, int num_ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
  cfg.blockDim = dim3(kSwaThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fmha_swa_kernel<BF16, NORM>, tq, tk, tv, to, a);
}

}  // namespace

const void* const kSwaKernels[4] = {
    reinterpret_cast<const void*>(fmha_swa_kernel<false, false>), reinterpret_cast<const void*>(fmha_swa_kernel<true, false>),
    reinterpret_cast<const void*>(fmha_swa_kernel<false, true>), reinterpret_cast<const void*>(fmha_swa_kernel<true, true>)};

cudaError_t fmha_swa_set_attributes() {
  for (const void* f : kSwaKernels) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool fmha_swa_check() {
  for (const void* f : kSwaKernels) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, f) != cudaSuccess || attr.binaryVersion != 103) return false;
  }
  return true;
}

cudaError_t fmha_swa_launch(bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const FmhaSwaArgs& a, int num_ctas, cudaStream_t stream) {
  if (a.qk_norm)
    return bf16 ? launch<true, true>(tq, tk, tv, to, a, num_ctas, stream)
                : launch<false, true>(tq, tk, tv, to, a, num_ctas, stream);
  return bf16 ? launch<true, false>(tq, tk, tv, to, a, num_ctas, stream)
              : launch<false, false>(tq, tk, tv, to, a, num_ctas, stream);
}

}  // namespace sa
