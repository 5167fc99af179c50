// sa_fmha.cu -- fused attention on rotated q', k' for sm_103a (GB300).
//
// Computes out = softmax(q' k'^T / sqrt(d)) v with the softmax accumulated in FP32
// (HF discussion #3 "fp16mixed attention-core fix", section "The bug": SDPA on fp16 inputs,
// FMHA accumulating the softmax in FP32), its differential form
// out = O(Q1,K1) - lambda_h * O(Q2,K2) with the subtraction done in FP32 on the FP32
// accumulators (HF discussion #6 "sm_120 SAME-L", section "How the kernels differ"), and the
// symmetric sliding window |i - j| <= w (same page, "Three gotchas").
//
// One CTA (384 threads, 1 per SM) owns one unit: 256 query rows of one (batch, head) as two
// 128-row tiles (standard), or 128 rows with both maps (differential).  Warp roles:
//   warps 0-3, 4-7  softmax warpgroups, one per tile / map (stream s): thread = query row =
//                   TMEM lane; with a raw q they first rotate their Q row in shared memory
//                   (RoPE prologue, from the RoPE pass's FP32 (cos, sin) table).
//   warp 8          TMA producer of Q and of the K ring (128 keys per stage); in the standard
//                   kernel also the issuer of both streams' S MMAs.
//   warp 9          TMEM allocator and the MMA issuer of stream 0 (P.V only, standard kernel).
//   warp 10         the MMA issuer of stream 1 (likewise).
//   warp 11         TMA producer of the V ring.
// Per K/V tile and stream s:
//   S_s = Q_s K^T      tcgen05.mma, A and B from 128B-swizzled smem, fp32 into TMEM
//   P_s = exp2(S_s*c - m)   softmax warps: tcgen05.ld S, row max, lazy rescale of O_s
//                      (only when the running max grows by more than 2^8), fp16/bf16 P
//                      written to TMEM (standard) or to shared memory (differential)
//   O_s += P_s V       tcgen05.mma, A = P from TMEM or smem, B = V (MN-major) from smem
// In the differential kernel the two warpgroups take turns on the exponential phase.  Each
// stream's S buffer is released as soon as the softmax warps hold S in registers, so the next
// S MMA overlaps the softmax.
// TMEM (512 columns): standard S0|S1|P0|P1|O0|O1 = 128|128|64|64|64|64;
// differential S0|S1|O0|O1 = 128|128|128|128.
// The sliding window visits only the key tiles of [q0 - w, q_last + w], tiled from its first
// key; element masks are applied only on tiles that are not entirely inside every row's window.
// When the units leave the GPU's last wave partly empty, the tail units are cut into key-range
// pieces (one CTA each) whose FP32 partial results the last piece merges in a fixed order.
// Every wait is bounded: on timeout a warp sets the device error word and a CTA-wide abort
// flag, waits (bounded) for its own copies / MMAs in flight, and the CTA frees TMEM and exits.
#include <type_traits>

#include "sa_kernels.h"
#include "sa_pipe.cuh"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kTile = kBlockM * kHeadDim * 2;  // bytes of one 128 x 64 fp16/bf16 tile (16 KB)
constexpr int kTmaWarp = 8;   // TMA producer of Q and the K ring
constexpr int kMmaWarp = 9;    // first MMA issuer (stream 0); also allocates TMEM
                               // (warp 10: the MMA issuer of stream 1)
constexpr int kTmaWarpV = 11;  // TMA producer of the V ring
constexpr uint32_t kTmemCols = 512;

template <bool DIFF>
struct Cfg {
  // K and V have rings of their own: a K stage is free again as soon as the S MMAs that read it
  // are done, a V stage once the P.V MMAs are, so each K tile can be fetched well ahead of use.
  static constexpr int NSK = DIFF ? 2 : 4;                      // K ring stages
  static constexpr int NSV = DIFF ? 2 : 4;                      // V ring stages
  static constexpr int DV = DIFF ? 128 : 64;                    // value / output width
  static constexpr int ROWS = fmha_rows_per_cta(DIFF);          // query rows per CTA
  static constexpr int Q_BYTES = 2 * kTile;                     // two Q tiles (or maps)
  static constexpr int K_STAGE = DIFF ? 2 * kTile : kTile;      // K (both maps for DIFF)
  static constexpr int V_STAGE = DIFF ? 2 * kTile : kTile;      // V: 128 keys x DV
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * K_STAGE;
  // Differential only: P of both maps in shared memory (128 rows x 128 keys each, two
  // 64-key swizzle atoms), the A operand of an SS P.V MMA.
  static constexpr int P_BYTES = DIFF ? 4 * kTile : 0;
  static constexpr int OFF_P = OFF_V + NSV * V_STAGE;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  // barriers: q_full, q_ready[2], k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2],
  //           p_full[2], pv_done[2], s_free[2], o_full[2], drain[2], turn[2][4], drain_k
  static constexpr int NBAR = 1 + 2 + 2 * NSK + 2 * NSV + 2 + 2 + 2 + 2 + 2 + 2 + 8 + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;           // tmem base, abort flag, ticket
  static constexpr int OFF_LSUM = OFF_MISC + 16;                // float [2][128]
  static constexpr int SMEM_USED = OFF_LSUM + 2 * kBlockM * 4;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;           // slack for 1 KB alignment
  __device__ static uint32_t s_col(int s) { return s * 128; }
  __device__ static uint32_t p_col(int s) { return 256 + s * 64; }   // standard only
  __device__ static uint32_t o_col(int s) { return DIFF ? 256 + s * 128 : 384 + s * 64; }
};

static_assert(Cfg<false>::SMEM_ALLOC <= 227 * 1024, "smem budget");
static_assert(Cfg<true>::SMEM_ALLOC <= 227 * 1024, "smem budget");
static_assert(Cfg<false>::SMEM_USED > 114 * 1024, "one CTA per SM keeps TMEM allocation uncontended");

struct Barriers {
  uint32_t q_full, q_ready0, k_full0, k_empty0, v_full0, v_empty0, s_full0, p_full0, pv_done0, s_free0, o_full0,
      drain0, turn0;
  // the S MMAs of the standard kernel's K producer warp have completed (before TMEM is released)
  uint32_t drain_k;
  __device__ uint32_t q_ready(int s) const { return q_ready0 + 8 * s; }
  __device__ uint32_t k_full(int i) const { return k_full0 + 8 * i; }
  __device__ uint32_t k_empty(int i) const { return k_empty0 + 8 * i; }
  __device__ uint32_t v_full(int i) const { return v_full0 + 8 * i; }
  __device__ uint32_t v_empty(int i) const { return v_empty0 + 8 * i; }
  __device__ uint32_t s_full(int s) const { return s_full0 + 8 * s; }
  __device__ uint32_t p_full(int s) const { return p_full0 + 8 * s; }
  __device__ uint32_t pv_done(int s) const { return pv_done0 + 8 * s; }
  __device__ uint32_t s_free(int s) const { return s_free0 + 8 * s; }
  __device__ uint32_t o_full(int s) const { return o_full0 + 8 * s; }
  __device__ uint32_t drain(int s) const { return drain0 + 8 * s; }
  // exp-phase turn of warpgroup s on SM sub-partition q (warps q and q + 4 share it)
  __device__ uint32_t turn(int s, int q) const { return turn0 + 8 * (4 * s + q); }
};

// This CTA's index, read from the special register each time (not a value the compiler keeps).
__device__ __forceinline__ unsigned cta_index() {
  unsigned x;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(x));
  return x;
}

// Counts one finished piece of a unit in this launch; true for the piece that completes the
// unit.  The counter's upper half holds the launch's epoch (never 0), so a value left by an
// earlier launch starts a fresh count; the last piece also clears the counter, so that a
// replay of the same launch (a CUDA graph keeps its epoch) starts fresh too.
__device__ bool take_ticket(unsigned long long* cnt, unsigned epoch, int npieces) {
  const unsigned long long tag = static_cast<unsigned long long>(epoch) << 32;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cnt), assumed;
  do {
    assumed = old;
    const unsigned long long nv = (assumed >> 32) == epoch ? assumed + 1 : (tag | 1ull);
    old = atomicCAS(cnt, assumed, nv);
  } while (old != assumed);
  const unsigned long long mine = (old >> 32) == epoch ? (old & 0xffffffffull) + 1 : 1ull;
  if (mine != static_cast<unsigned long long>(npieces)) return false;
  atomicExch(cnt, 0ull);
  return true;
}

// RoPE prologue of one Q row (thread r of a softmax warpgroup): the TMA brought the tile in
// raw; the row is rotated in place (128-byte-swizzled smem: 16-byte chunk c of row r sits at
// c ^ (r & 7)), pairs [8g, 8g + 8) from chunks g and g + 4, with the RoPE pass's FP32
// (cos, sin) of the row's position and the pre-pass's arithmetic.  With gamma (NORM) the row is
// QK-RMS-normalised first, with the pre-pass's sum order and scaling, so its bits again equal
// the pre-pass's.  Kept out of line so that its registers do not weigh on the softmax loop's.
// Returns the warp-uniform wait outcome.
template <bool BF16, bool NORM>
__device__ __noinline__ bool q_rope_prologue(const float2* cs, int cs_stride, bool cs_static, int L, int grow,
                                             uint32_t row, int r, uint32_t q_full, volatile int* abort_flag,
                                             int* err, uint64_t tmo, const float* gamma, float eps) {
  // a per-call table is the RoPE pass's output: wait for that grid (programmatic dependent
  // launch); the handle's table was written long before
  if (!cs_static) asm volatile("griddepcontrol.wait;" ::: "memory");
  // the row's (cos, sin) pairs ([16][cs_stride] float4 table: a warp's loads are contiguous),
  // loaded while the TMA brings Q
  float4 t[16];
  const float4* cs4 = reinterpret_cast<const float4*>(cs) + min(grow, L - 1);
#pragma unroll
  for (int m = 0; m < 16; ++m) t[m] = __ldg(cs4 + static_cast<size_t>(m) * cs_stride);
  bool ok = pwait(q_full, 0, abort_flag, err, kErrSoftmax, tmo);
  ok = __all_sync(0xffffffffu, ok);
  if (ok && grow < L) {
    uint4 lo[4], hi[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      lo[g] = ld_shared_v4(row + ((g ^ (r & 7)) << 4));
      hi[g] = ld_shared_v4(row + (((g + 4) ^ (r & 7)) << 4));
    }
    float inv = 1.0f;
    if (NORM) {
      float tg[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) tg[g] = sumsq8<BF16>(lo[g]) + sumsq8<BF16>(hi[g]);
      inv = qknorm_inv_rms((tg[0] + tg[1]) + (tg[2] + tg[3]), eps);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float cg[8], sg[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cg[2 * i] = t[4 * g + i].x;
        cg[2 * i + 1] = t[4 * g + i].y;
        sg[2 * i] = t[4 * g + i].z;
        sg[2 * i + 1] = t[4 * g + i].w;
      }
      uint4 olo, ohi;
      if (NORM) {
        float sl[8], sh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          sl[i] = __fmul_rn(inv, gamma[8 * g + i]);
          sh[i] = __fmul_rn(inv, gamma[32 + 8 * g + i]);
        }
        rope_rotate8_scaled<BF16>(lo[g], hi[g], cg, sg, sl, sh, olo, ohi);
      } else {
        rope_rotate8<BF16>(lo[g], hi[g], cg, sg, olo, ohi);
      }
      const uint32_t a_lo = row + ((g ^ (r & 7)) << 4), a_hi = row + (((g + 4) ^ (r & 7)) << 4);
      st_shared_v4(a_lo, olo.x, olo.y, olo.z, olo.w);
      st_shared_v4(a_hi, ohi.x, ohi.y, ohi.z, ohi.w);
    }
  }
  return ok;
}

// O_s *= f in TMEM, the lazy rescale.  It is rare, and kept out of line it adds no code to the
// softmax loop (whose speed depends on its size: the loop is close to the instruction cache's
// capacity).
template <int DV>
__device__ __noinline__ void rescale_o(uint32_t taddr, float f) {
#pragma unroll
  for (int cc = 0; cc < DV / 32; ++cc) {
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

// Key masking a launch needs, a template parameter because the softmax loop's speed depends on
// its code size (the loop is close to the instruction cache's capacity): none (full attention,
// L a multiple of 128), the sequence tail (full attention, the last key tile crosses L), or the
// window (and the tail).
constexpr int kMaskNone = 0, kMaskTail = 1, kMaskWindow = 2;

// One key tile of a softmax warp (tile `it` of its unit, stream s): wait for S, load it and
// release it, mask it (TMASK: none; the sequence tail, columns >= j_hi; or, when need_mask,
// the window, columns outside [j_lo, j_hi)), row max and lazy rescale, exponentials on this
// warp's turn, row sum, P stored for its P.V MMA.  Returns the warp-uniform wait outcome.
template <bool DIFF, bool BF16, int TMASK>
__device__ __forceinline__ bool softmax_tile(const Barriers& bar, int it, uint32_t tmem, uint32_t lane_off,
                                             int s, int quarter, int lane, int r, uint32_t sP, float c,
                                             float tau, bool need_mask, int j_lo, int j_hi, float& m_use,
                                             float& l_sum, volatile int* abort_flag, int* err, uint64_t tmo) {
  using C = Cfg<DIFF>;
  bool ok;
  ok = pwait(bar.s_full(s), it & 1, abort_flag, err, kErrSoftmax, tmo);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  tc_fence_after();
  // S row and its maximum in one load: the tensor memory's reducing load (sm_103a) returns the
  // max of the 128 values with them, so an unmasked tile spends no instruction on its row max.
  uint32_t sr[kBlockN];
  float mt;
  tmem_ld128_max_nowait(tmem + C::s_col(s) + lane_off, sr, mt);
  tmem_wait_ld_128_max(sr, mt);
  {
    // S_s is in registers: the issuer may write the next S_s into these columns now.
    // Every lane has waited for its own load; after the warp sync one lane arrives.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.s_free(s));
  }

  if (TMASK == kMaskTail || (TMASK == kMaskWindow && need_mask)) {
    // this row's valid keys are columns [j_lo, j_hi) of the tile (one compare per column
    // against bounds computed once keeps the masking code short); the loaded maximum also
    // covers the masked columns, so the row max is taken again over the masked row.
#pragma unroll
    for (int j = 0; j < kBlockN; ++j)
      if (j >= j_hi || (TMASK == kMaskWindow && j < j_lo)) sr[j] = __float_as_uint(-INFINITY);
    // 8 independent chains; chain q covers elements q, q + 8, ..., q + 120.
    float mx[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) mx[q] = fmaxf(__uint_as_float(sr[q]), __uint_as_float(sr[q + 8]));
#pragma unroll
    for (int j = 16; j < kBlockN; j += 16) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        mx[q] = fmax3(mx[q], __uint_as_float(sr[j + q]), __uint_as_float(sr[j + 8 + q]));
    }
    mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
  }

  // Lazy rescale: keep the old running max unless this tile raises it by more than tau
  // (P then stays <= 2^8).  The decision is warp-uniform because tcgen05.ld/st are.
  float f = 1.0f;
  bool rescale = false;
  if (it == 0) {
    m_use = mt;
  } else if (__any_sync(0xffffffffu, mt > m_use + tau)) {
    const float m_new = fmaxf(m_use, mt);
    f = (m_new == m_use) ? 1.0f : ex2_approx((m_use - m_new) * c);
    m_use = m_new;
    rescale = true;
  }
  const float mb = (m_use == -INFINITY) ? 0.0f : m_use * c;
  const float2 c2 = make_float2(c, c), nmb2 = make_float2(-mb, -mb);
  if (DIFF) {
    // the differential kernel's warps take turns on the exp unit (see the kernel's softmax part)
    ok = pwait(bar.turn(s, quarter), it & 1, abort_flag, err, kErrSoftmax, tmo);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
  }
  // Exponentials of the whole row into registers (packed pairs): P_s(it) is computed
  // before the wait for P_s V(it - 1), which has the whole exponential phase to finish.
  float2 sum0 = make_float2(0.0f, 0.0f), sum1 = make_float2(0.0f, 0.0f);
  uint32_t pk[kBlockN / 2];
#pragma unroll
  for (int j = 0; j < kBlockN / 2; j += 2) {
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
  if (DIFF) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.turn(1 - s, quarter));
  }
  const float2 sum = fadd2(sum0, sum1);
  l_sum = fmaf(l_sum, f, sum.x + sum.y);
  if (it > 0) {
    // P_s and O_s are still read / written by P_s V of the previous tile until it is done.
    ok = pwait(bar.pv_done(s), (it - 1) & 1, abort_flag, err, kErrSoftmax, tmo);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    tc_fence_after();
  }
  if (DIFF) {
    // row r of the K-major, 128-byte-swizzled P tile: atom h (keys 64h..64h+63),
    // 16-byte chunk kq lands at chunk kq ^ (r & 7)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t row_base = sP + s * 2 * kTile + h * kTile + r * 128;
#pragma unroll
      for (int kq = 0; kq < 8; ++kq)
        st_shared_v4(row_base + ((kq ^ (r & 7)) << 4), pk[32 * h + 4 * kq], pk[32 * h + 4 * kq + 1],
                     pk[32 * h + 4 * kq + 2], pk[32 * h + 4 * kq + 3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    tmem_st32(tmem + C::p_col(s) + lane_off, pk);
    tmem_st32(tmem + C::p_col(s) + lane_off + 32, pk + 32);
  }
  if (rescale) rescale_o<C::DV>(tmem + C::o_col(s) + lane_off, f);
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar.p_full(s));
  return true;
}

template <bool DIFF, bool BF16, int MASK>
__global__ void __launch_bounds__(kFmhaThreads, 1)
    fmha_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FmhaArgs a) {
  using C = Cfg<DIFF>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sP = sb + C::OFF_P;

  Barriers bar;
  bar.q_full = sb + C::OFF_BAR;
  bar.q_ready0 = bar.q_full + 8;
  bar.k_full0 = bar.q_ready0 + 16;
  bar.k_empty0 = bar.k_full0 + 8 * C::NSK;
  bar.v_full0 = bar.k_empty0 + 8 * C::NSK;
  bar.v_empty0 = bar.v_full0 + 8 * C::NSV;
  bar.s_full0 = bar.v_empty0 + 8 * C::NSV;
  bar.p_full0 = bar.s_full0 + 16;
  bar.pv_done0 = bar.p_full0 + 16;
  bar.s_free0 = bar.pv_done0 + 16;
  bar.o_full0 = bar.s_free0 + 16;
  bar.drain0 = bar.o_full0 + 16;
  bar.turn0 = bar.drain0 + 16;
  bar.drain_k = bar.turn0 + 64;

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* ticket = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  float* lsum = reinterpret_cast<float*>(smem + C::OFF_LSUM);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = a.L;
  // The unit of this CTA: a whole one, or a piece (a share of the key tiles) of a tail unit.
  const bool piece = static_cast<int>(blockIdx.x) >= a.whole_ctas;
  const int pidx = static_cast<int>(blockIdx.x) - a.whole_ctas;   // piece index (pieces only)
  const int unit = piece ? a.whole_ctas + pidx / a.tail_k : static_cast<int>(blockIdx.x);
  const int bh = unit / a.n_qblocks;
  const int q0 = (unit % a.n_qblocks) * C::ROWS;
  const int q_last = min(L, q0 + C::ROWS) - 1;
  const int w = a.window;

  // K/V tiles this CTA visits.
  // Keys [k_first, k_first + 128 n) in 128-key tiles: all keys, or the unit's window span
  // [q0 - w, q_last + w] clipped to [0, L - 1], tiled from its first key (a TMA box may start at
  // any row), which visits ceil(span / 128) tiles rather than every 128-aligned tile it touches.
  int k_first = 0, t_lo = 0, t_hi = (L - 1) / kBlockN;
  if (w >= 0) {
    k_first = max(0, q0 - w);
    t_hi = (min(L - 1, q_last + w) - k_first) / kBlockN;
  }
  if (piece) {
    // piece k of tail_k: tiles [t_lo + k nt / tail_k, t_lo + (k + 1) nt / tail_k), never empty
    // (the host keeps tail_k <= nt)
    const int nt = t_hi - t_lo + 1, k = pidx % a.tail_k;
    t_hi = t_lo + (k + 1) * nt / a.tail_k - 1;
    t_lo = t_lo + k * nt / a.tail_k;
  }
  const int n_tiles = t_hi - t_lo + 1;
  const uint64_t tmo = a.timeout_ns;
  // Waits for work already in flight (copies, MMAs) before shared memory / TMEM are released
  // always get at least a second, whatever the pipeline limit is.
  const uint64_t drain_tmo = tmo > 1000000000ull ? tmo : 1000000000ull;

  if (threadIdx.x == 0) {
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < 2; ++s) mbar_init(bar.q_ready(s), 4);   // one arrival per softmax warp
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(bar.k_full(i), 1);
      mbar_init(bar.k_empty(i), 2);    // one commit per stream's S MMAs
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(bar.v_full(i), 1);
      mbar_init(bar.v_empty(i), 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.s_full(s), 1);
      mbar_init(bar.p_full(s), 4);       // one elected arrival per softmax warp
      mbar_init(bar.pv_done(s), 1);
      mbar_init(bar.s_free(s), 4);
      mbar_init(bar.o_full(s), 1);
      mbar_init(bar.drain(s), 1);
      for (int q = 0; q < 4; ++q) mbar_init(bar.turn(s, q), 1);
    }
    mbar_init(bar.drain_k, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
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

  if (warp >= 8) {
  // Control warpgroup: K producer, the two MMA issuers, V producer; few registers.  These warps
  // run warp-uniform code: every lane waits on the barriers and one lane, elected inside each
  // issuing instruction, issues the copies / MMAs / commits (the operands stay warp-uniform,
  // which keeps the issue of each tcgen05.mma short).
  // the standard kernel's register split (the differential kernel runs without one)
  if (!DIFF) regs_dec<kControlRegs>();
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ K producer (+ Q)
    // This grid may have been started early (programmatic dependent launch) while the kernel
    // before it on the stream (the RoPE pass, which writes q', k') is still running: wait for
    // it before the first load.
    // Raw q (the Q prologue case) is not written by the RoPE pass: load it, and warm L2 with the
    // Q tiles of the CTA one wave later, before that wait.
    const bool raw_q = a.cs != nullptr;
    if (!raw_q) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int plane_q = DIFF ? 2 * bh : bh;
    mbar_arrive_expect_tx_w(bar.q_full, C::Q_BYTES);
    if (DIFF) {
      tma_load_3d_w(sQ, &tm_q, bar.q_full, 0, q0, plane_q);
      tma_load_3d_w(sQ + kTile, &tm_q, bar.q_full, 0, q0, plane_q + 1);
    } else {
      tma_load_3d_w(sQ, &tm_q, bar.q_full, 0, q0, plane_q);
      tma_load_3d_w(sQ + kTile, &tm_q, bar.q_full, 0, q0 + kBlockM, plane_q);
    }
    if (raw_q) {
      const int c2 = static_cast<int>(blockIdx.x) + a.wave;
      if (a.wave > 0 && c2 < static_cast<int>(gridDim.x) && lane == 0) {
        const int u2 = c2 >= a.whole_ctas ? a.whole_ctas + (c2 - a.whole_ctas) / a.tail_k : c2;
        const int bh2 = u2 / a.n_qblocks, q02 = (u2 % a.n_qblocks) * C::ROWS;
        tma_prefetch_l2_3d(&tm_q, 0, q02, DIFF ? 2 * bh2 : bh2);
        tma_prefetch_l2_3d(&tm_q, 0, DIFF ? q02 : q02 + kBlockM, DIFF ? 2 * bh2 + 1 : bh2);
      }
      __syncwarp();
      asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    int issued = 0;
    auto load_k = [&](int it) {
      const int st = it % C::NSK;
      if (!pwait_w(bar.k_empty(st), ((it / C::NSK) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo))
        return false;
      const int key0 = k_first + (t_lo + it) * kBlockN;
      const uint32_t k_dst = sK + st * C::K_STAGE;
      mbar_arrive_expect_tx_w(bar.k_full(st), C::K_STAGE);
      if (DIFF) {
        tma_load_3d_w(k_dst, &tm_k, bar.k_full(st), 0, key0, 2 * bh);
        tma_load_3d_w(k_dst + kTile, &tm_k, bar.k_full(st), 0, key0, 2 * bh + 1);
      } else {
        tma_load_3d_w(k_dst, &tm_k, bar.k_full(st), 0, key0, bh);
      }
      issued = it + 1;
      return true;
    };
    if constexpr (DIFF) {
      for (int it = 0; it < n_tiles; ++it)
        if (!load_k(it)) break;
    } else {
      // The standard kernel's K producer also issues both streams' S MMAs (the MMA issuers keep
      // the P.V MMAs): each SM sub-partition that hosts an issuing warp gives some of its issue
      // slots to it, and its softmax warps then finish their tiles last, so the issue work is
      // spread over three sub-partitions instead of two.  Per tile: S_0(j) and S_1(j), each once
      // the softmax warps hold S_s(j - 1) in registers (S is single-buffered per stream), then
      // K(j + NSK - 1) into the stage that S(j - 1) has released.
      constexpr uint32_t idesc_s = make_idesc_f16(kBlockM, kBlockN, BF16, false);
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sQ + kTile, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      const uint32_t q_bar0 = raw_q ? bar.q_ready(0) : bar.q_full;
      const uint32_t q_bar1 = raw_q ? bar.q_ready(1) : bar.q_full;
      constexpr int eb = kErrMma;
      bool ok = true;
      for (int it = 0; ok && it < C::NSK - 1 && it < n_tiles; ++it) ok = load_k(it);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % C::NSK;
        const uint64_t dk = dk0 + static_cast<uint64_t>(st * (C::K_STAGE >> 4));
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          ok = pwait_w(j == 0 ? (s == 0 ? q_bar0 : q_bar1) : bar.s_free(s), j == 0 ? 0u : static_cast<uint32_t>((j - 1) & 1),
                       abort_flag, a.err, eb, tmo) &&
               pwait_w(bar.k_full(st), (j / C::NSK) & 1, abort_flag, a.err, eb, tmo);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = s == 0 ? dq0 : dq1;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            umma_ss_w(tmem + C::s_col(s), dq + 2 * kk, dk + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
          umma_commit_w(bar.s_full(s));
          umma_commit_w(bar.k_empty(st));
        }
        if (ok && j + C::NSK - 1 < n_tiles) ok = load_k(j + C::NSK - 1);
      }
      // no S MMA of this warp may still be running when TMEM is released
      umma_commit_w(bar.drain_k);
      mbar_wait_limit(bar.drain_k, 0, drain_tmo);
    }
    // Let the copies already issued land before the CTA's shared memory goes away (after a
    // normal run these phases have completed and the waits return at once).
    mbar_wait_limit(bar.q_full, 0, drain_tmo);
    for (int it = issued > C::NSK ? issued - C::NSK : 0; it < issued; ++it)
      mbar_wait_limit(bar.k_full(it % C::NSK), (it / C::NSK) & 1, drain_tmo);
    __syncwarp();
  } else if (warp == kTmaWarpV) {
    // ------------------------------------------------------------------ V producer
    // v is not written by the RoPE pass, and the work before that pass on the stream has
    // completed once this grid runs: no wait on the grid dependency.
    int issued = 0;
    for (int it = 0; it < n_tiles; ++it) {
      const int st = it % C::NSV;
      if (!pwait_w(bar.v_empty(st), ((it / C::NSV) & 1) ^ 1, abort_flag, a.err, kErrProducer, tmo))
        break;
      const int key0 = k_first + (t_lo + it) * kBlockN;
      const uint32_t v_dst = sV + st * C::V_STAGE;
      mbar_arrive_expect_tx_w(bar.v_full(st), C::V_STAGE);
      tma_load_3d_w(v_dst, &tm_v, bar.v_full(st), 0, key0, bh);
      if (DIFF) tma_load_3d_w(v_dst + kTile, &tm_v, bar.v_full(st), 64, key0, bh);
      issued = it + 1;
    }
    for (int it = issued > C::NSV ? issued - C::NSV : 0; it < issued; ++it)
      mbar_wait_limit(bar.v_full(it % C::NSV), (it / C::NSV) & 1, drain_tmo);
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ MMA issuers
    // One issuing warp per stream s (query tile s, or map s).  Differential kernel: after the
    // prologue each issues, per tile, one block: P.V_s(i) as soon as P_s(i) is ready, then
    // S_s(i + 2) (it overwrites S_s(i + 1), which the softmax warps load right after P_s(i)).
    // Standard kernel: P.V_s(i) only (the K producer issues the S MMAs; P has TMEM columns of
    // its own, so no S MMA can overwrite a P that a P.V MMA has yet to read).  The stream index
    // is a compile-time constant in each instance so that every operand is warp-uniform.
    auto issuer = [&](auto stream) {
      constexpr int s = decltype(stream)::value;
      constexpr uint32_t idesc_s = make_idesc_f16(kBlockM, kBlockN, BF16, false);
      constexpr uint32_t idesc_o = make_idesc_f16(kBlockM, C::DV, BF16, true);
      // Descriptors computed once; the 14-bit address field advances by constant steps
      // (32 B along K inside a swizzle row, 2 KB per 16 keys of V, one stage per ring slot).
      const uint64_t dq = smem_desc_sw128(sQ + s * kTile, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK + (DIFF ? s * kTile : 0), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sV, kTile, 1024);
      const uint32_t d_s = tmem + C::s_col(s), d_o = tmem + C::o_col(s), a_p = tmem + C::p_col(s);
      // differential: P_s in shared memory, two 64-key atoms of 16 KB (K-major, 128 B swizzle)
      const uint64_t dp0 = smem_desc_sw128(sP + s * 2 * kTile, 16, 1024);
      constexpr int eb = kErrMma;
      auto wait_k = [&](int it) {
        return pwait_w(bar.k_full(it % C::NSK), (it / C::NSK) & 1, abort_flag, a.err, eb, tmo);
      };
      auto issue_s = [&](int it) {
        const int st = it % C::NSK;
        const uint64_t dk = dk0 + static_cast<uint64_t>(st * (C::K_STAGE >> 4));
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          umma_ss_w(d_s, dq + 2 * kk, dk + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
        umma_commit_w(bar.s_full(s));
        umma_commit_w(bar.k_empty(st));
      };
      // Q tile s as the MMA reads it: straight from the TMA, or after the softmax warps' RoPE
      const uint32_t q_bar = a.cs != nullptr ? bar.q_ready(s) : bar.q_full;
      bool ok = true;
      if constexpr (DIFF) {
        ok = pwait_w(q_bar, 0, abort_flag, a.err, eb, tmo) && wait_k(0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
      }
      if (DIFF && ok && n_tiles > 1) {
        // S_s(1) once the softmax warps hold S_s(0) in registers
        ok = pwait_w(bar.s_free(s), 0, abort_flag, a.err, eb, tmo) && wait_k(1);
        if (ok) {
          tc_fence_after();
          issue_s(1);
        }
      }
      for (int it = 0; ok && it < n_tiles; ++it) {
        const int sv = it % C::NSV;
        // V(it) arrived long ago in the steady state: check it before waiting for P
        ok = pwait_w(bar.v_full(sv), (it / C::NSV) & 1, abort_flag, a.err, eb, tmo) &&
             pwait_w(bar.p_full(s), it & 1, abort_flag, a.err, eb, tmo);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(sv * (C::V_STAGE >> 4));
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          if (DIFF)
            umma_ss_w(d_o, dp0 + (kk >> 2) * (kTile >> 4) + 2 * (kk & 3), dv + 128 * kk, idesc_o, acc);
          else
            umma_ts_w(d_o, a_p + 8 * kk, dv + 128 * kk, idesc_o, acc);
        }
        umma_commit_w(bar.pv_done(s));
        umma_commit_w(bar.v_empty(sv));
        if (it + 1 == n_tiles) umma_commit_w(bar.o_full(s));
        if (DIFF && it + 2 < n_tiles) {
          ok = pwait_w(bar.s_free(s), (it + 1) & 1, abort_flag, a.err, eb, tmo) && wait_k(it + 2);
          if (!ok) break;
          tc_fence_after();
          issue_s(it + 2);
        }
      }
      // No MMA of this issuer may still be running when TMEM is released.
      umma_commit_w(bar.drain(s));
      mbar_wait_limit(bar.drain(s), 0, drain_tmo);
      __syncwarp();
    };
    if (warp == kMmaWarp)
      issuer(std::integral_constant<int, 0>{});
    else
      issuer(std::integral_constant<int, 1>{});
  }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    if (!DIFF) regs_inc<kSoftmaxRegs>();
    const int s = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                     // TMEM lane = tile row
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int grow = DIFF ? q0 + r : q0 + s * kBlockM + r;  // query row in the sequence
    const float c = a.scale_log2;
    const float tau = 8.0f / c;                            // lazy-rescale threshold (raw units)
    const int rows_lo = q0, rows_hi = q0 + C::ROWS - 1;
    float m_use = -INFINITY;
    float l_sum = 0.0f;
    bool ok = true;
    // Differential kernel: the two warpgroups take turns on the exponential phase, pairwise
    // per SM sub-partition (warp q of group 0 with warp q of group 1, which share one): group 0
    // goes first, each warp hands the turn to its partner when its exponentials are issued, so
    // one warp's TMEM / barrier / shared-memory work overlaps the other's exponentials.  The
    // standard kernel (d_v = 64, P in tensor memory, row max from the reducing load) runs
    // without turns: there the hand-over cost more than it saved (measured 8% at L = 4096).
    if (DIFF && s == 1 && lane == 0) mbar_arrive(bar.turn(0, quarter));

    if (a.cs != nullptr) {
      // RoPE prologue on this warpgroup's Q tile, then the tile goes to its MMA issuer.
      if (a.qk_norm)
        ok = q_rope_prologue<BF16, true>(a.cs, a.cs_stride, a.cs_static, L, grow, sQ + s * kTile + r * 128, r,
                                         bar.q_full, abort_flag, a.err, tmo, a.gamma_q, a.eps);
      else
        ok = q_rope_prologue<BF16, false>(a.cs, a.cs_stride, a.cs_static, L, grow, sQ + s * kTile + r * 128, r,
                                          bar.q_full, abort_flag, a.err, tmo, nullptr, 0.0f);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.q_ready(s));
    }

    // The tile that crosses the end of the sequence (the unit's last, if any) is peeled off the
    // loop in the tail-masked kernel, so the loop body holds no masking code.
    const bool peel_tail = MASK == kMaskTail && k_first + (t_lo + n_tiles) * kBlockN > L;
    const int n_loop = n_tiles - (peel_tail ? 1 : 0);
    for (int it = 0; it < n_loop; ++it) {
      if (MASK != kMaskWindow) {
        ok = softmax_tile<DIFF, BF16, kMaskNone>(bar, it, tmem, lane_off, s, quarter, lane, r, sP, c, tau, false,
                                                 0, 0, m_use, l_sum, abort_flag, a.err, tmo);
      } else {
        const int key0 = k_first + (t_lo + it) * kBlockN;
        const bool need_mask =
            (key0 + kBlockN > L) || !(key0 >= rows_hi - w && key0 + kBlockN - 1 <= rows_lo + w);
        ok = softmax_tile<DIFF, BF16, kMaskWindow>(bar, it, tmem, lane_off, s, quarter, lane, r, sP, c, tau,
                                                   need_mask, grow - w - key0,
                                                   min(L - key0, grow + w + 1 - key0), m_use, l_sum,
                                                   abort_flag, a.err, tmo);
      }
      if (!ok) break;
    }
    if (peel_tail && ok)
      ok = softmax_tile<DIFF, BF16, kMaskTail>(bar, n_loop, tmem, lane_off, s, quarter, lane, r, sP, c, tau, true,
                                               0, L - (k_first + (t_lo + n_loop) * kBlockN), m_use, l_sum,
                                               abort_flag, a.err, tmo);

    // ---------------------------------------------------------------- epilogue
    if (ok) ok = pwait(bar.o_full(s), 0, abort_flag, a.err, kErrSoftmax, tmo);
    if (DIFF && ok) ok = pwait(bar.o_full(1 - s), 0, abort_flag, a.err, kErrSoftmax, tmo);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    bool write_out = true;
    // The piece index is read again here rather than kept live through the loop (registers are
    // the softmax warps' scarce resource there).
    const int pidx_e = static_cast<int>(cta_index()) - a.whole_ctas;
    if (pidx_e >= 0) {
      // A piece of a tail unit: store its un-normalised O, running max (raw score units) and row
      // sum; the piece that finishes last merges all of the unit's pieces, in piece order, into
      // O_s in TMEM and l_sum, and writes the output below as for a whole unit.  A slot holds O
      // as [d_v / 4][256 rows] float4 (a warp's access is 512 contiguous bytes), then the
      // running maxima [256] and the row sums [256].
      constexpr int PF = fmha_partial_floats(DIFF);
      constexpr int NR = 2 * kBlockM;                    // rows of a slot (both streams)
      const size_t row_off = static_cast<size_t>(s * kBlockM + r);
      float* part = a.partials + static_cast<size_t>(pidx_e) * PF;
      if (ok) {
        float4* d4 = reinterpret_cast<float4*>(part) + row_off;
#pragma unroll
        for (int cc = 0; cc < C::DV / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32_nowait(tmem + C::o_col(s) + lane_off + 32 * cc, o);
          tmem_wait_ld_32(o);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[(8 * cc + q) * NR] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                                __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
        }
        part[2 * kBlockM * C::DV + row_off] = m_use;
        part[2 * kBlockM * C::DV + 2 * kBlockM + row_off] = l_sum;
      }
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (threadIdx.x == 0)
        *ticket = take_ticket(a.counters + a.whole_ctas + pidx_e / a.tail_k, a.epoch, a.tail_k) ? 1 : 0;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      write_out = *ticket != 0;
      if (write_out) {
        // every other piece's stores are visible after this fence
        __threadfence();
        const int p0 = pidx_e - pidx_e % a.tail_k;
        const float* base = a.partials + static_cast<size_t>(p0) * PF;
        // Piece weights 2^((m_p - mm) c); a piece whose keys all lie outside this row's window
        // (m_p = -inf) contributes nothing.  Every load of a step is issued before its use.
        float mp[kMaxTailK], lp[kMaxTailK], wt[kMaxTailK];
#pragma unroll
        for (int i = 0; i < kMaxTailK; ++i) {
          mp[i] = i < a.tail_k ? __ldcg(base + i * PF + 2 * kBlockM * C::DV + row_off) : -INFINITY;
          lp[i] = i < a.tail_k ? __ldcg(base + i * PF + 2 * kBlockM * C::DV + 2 * kBlockM + row_off) : 0.0f;
        }
        float mm = mp[0];
#pragma unroll
        for (int i = 1; i < kMaxTailK; ++i) mm = fmaxf(mm, mp[i]);
        float lm = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxTailK; ++i) {
          wt[i] = mp[i] == -INFINITY ? 0.0f : ex2_approx((mp[i] - mm) * c);
          lm = fmaf(lp[i], wt[i], lm);
        }
        l_sum = lm;
        // the merged O, 32 columns at a time, goes back to TMEM for the output code below
#pragma unroll
        for (int cc = 0; cc < C::DV / 32; ++cc) {
          float4 v4[kMaxTailK][8];
#pragma unroll
          for (int i = 0; i < kMaxTailK; ++i) {
            const float4* po = reinterpret_cast<const float4*>(base + i * PF) + row_off;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              v4[i][q] = i < a.tail_k ? __ldcg(po + (8 * cc + q) * NR) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          uint32_t o[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kMaxTailK; ++i) {
              acc.x = fmaf(v4[i][q].x, wt[i], acc.x);
              acc.y = fmaf(v4[i][q].y, wt[i], acc.y);
              acc.z = fmaf(v4[i][q].z, wt[i], acc.z);
              acc.w = fmaf(v4[i][q].w, wt[i], acc.w);
            }
            o[4 * q] = __float_as_uint(acc.x);
            o[4 * q + 1] = __float_as_uint(acc.y);
            o[4 * q + 2] = __float_as_uint(acc.z);
            o[4 * q + 3] = __float_as_uint(acc.w);
          }
          tmem_st32(tmem + C::o_col(s) + lane_off + 32 * cc, o);
        }
        tmem_wait_st();
      }
    }
    if (!write_out) {
      // another piece of this unit writes its output
    } else if (!DIFF) {
      const float inv = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
      uint16_t* dst = static_cast<uint16_t*>(a.out) +
                      (static_cast<size_t>(bh) * L + grow) * static_cast<size_t>(C::DV);
      if (ok) {
#pragma unroll
        for (int cc = 0; cc < C::DV / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32_nowait(tmem + C::o_col(s) + lane_off + 32 * cc, o);
          tmem_wait_ld_32(o);
          uint32_t pkd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pkd[j] = pack2<BF16>(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
          if (grow < L) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              d4[j] = make_uint4(pkd[4 * j], pkd[4 * j + 1], pkd[4 * j + 2], pkd[4 * j + 3]);
          }
        }
      }
    } else {
      lsum[s * kBlockM + r] = l_sum;
      tc_fence_before();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      tc_fence_after();
      const float l0 = lsum[r], l1 = lsum[kBlockM + r];
      const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f;
      const float inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
      const float lam = a.lambda[bh % a.H];
      uint16_t* dst = static_cast<uint16_t*>(a.out) +
                      (static_cast<size_t>(bh) * L + grow) * static_cast<size_t>(C::DV) + 64 * s;
      if (ok) {
        // warpgroup s writes output columns [64 s, 64 s + 64)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t col = 64 * s + 32 * cc;
          uint32_t o0[32], o1[32];
          tmem_ld32_nowait(tmem + C::o_col(0) + lane_off + col, o0);
          tmem_ld32_nowait(tmem + C::o_col(1) + lane_off + col, o1);
          tmem_wait_ld_32(o0);
          tmem_wait_ld_32(o1);
          uint32_t pkd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float y0 = fmaf(-lam, __uint_as_float(o1[2 * j]) * inv1, __uint_as_float(o0[2 * j]) * inv0);
            const float y1 =
                fmaf(-lam, __uint_as_float(o1[2 * j + 1]) * inv1, __uint_as_float(o0[2 * j + 1]) * inv0);
            pkd[j] = pack2<BF16>(y0, y1);
          }
          if (grow < L) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              d4[j] = make_uint4(pkd[4 * j], pkd[4 * j + 1], pkd[4 * j + 2], pkd[4 * j + 3]);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool DIFF, bool BF16>
cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(fmha_kernel<DIFF, BF16, kMaskNone>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<DIFF>::SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fmha_kernel<DIFF, BF16, kMaskTail>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<DIFF>::SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fmha_kernel<DIFF, BF16, kMaskWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<DIFF>::SMEM_ALLOC);
  return e;
}

// Launched with programmatic stream serialization: the CTAs may start while the previous
// kernel on the stream (the RoPE pass) finishes; only the TMA warp waits for it.
template <bool DIFF, bool BF16, int MASK>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const FmhaArgs& a, long long num_ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
  cfg.blockDim = dim3(kFmhaThreads);
  cfg.dynamicSmemBytes = Cfg<DIFF>::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fmha_kernel<DIFF, BF16, MASK>, tq, tk, tv, a);
}

template <bool DIFF, bool BF16>
cudaError_t launch_masked(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FmhaArgs& a, long long num_ctas, cudaStream_t stream) {
  if (a.window >= 0) return launch<DIFF, BF16, kMaskWindow>(tq, tk, tv, a, num_ctas, stream);
  if (a.L % kBlockN != 0) return launch<DIFF, BF16, kMaskTail>(tq, tk, tv, a, num_ctas, stream);
  return launch<DIFF, BF16, kMaskNone>(tq, tk, tv, a, num_ctas, stream);
}

}  // namespace

bool fmha_check_registers(int* got) {
  const void* fns[12] = {
      reinterpret_cast<const void*>(fmha_kernel<false, false, kMaskNone>),
      reinterpret_cast<const void*>(fmha_kernel<false, true, kMaskNone>),
      reinterpret_cast<const void*>(fmha_kernel<true, false, kMaskNone>),
      reinterpret_cast<const void*>(fmha_kernel<true, true, kMaskNone>),
      reinterpret_cast<const void*>(fmha_kernel<false, false, kMaskTail>),
      reinterpret_cast<const void*>(fmha_kernel<false, true, kMaskTail>),
      reinterpret_cast<const void*>(fmha_kernel<true, false, kMaskTail>),
      reinterpret_cast<const void*>(fmha_kernel<true, true, kMaskTail>),
      reinterpret_cast<const void*>(fmha_kernel<false, false, kMaskWindow>),
      reinterpret_cast<const void*>(fmha_kernel<false, true, kMaskWindow>),
      reinterpret_cast<const void*>(fmha_kernel<true, false, kMaskWindow>),
      reinterpret_cast<const void*>(fmha_kernel<true, true, kMaskWindow>)};
  for (const void* f : fns) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, f) != cudaSuccess) return false;
    *got = attr.numRegs;
    if (attr.numRegs != kFmhaLaunchRegs) return false;
    // the library holds sm_103a code only
    if (attr.binaryVersion != 103) return false;
  }
  return true;
}

cudaError_t fmha_set_attributes() {
  cudaError_t e;
  if ((e = set_attr<false, false>()) != cudaSuccess) return e;
  if ((e = set_attr<false, true>()) != cudaSuccess) return e;
  if ((e = set_attr<true, false>()) != cudaSuccess) return e;
  return set_attr<true, true>();
}

cudaError_t fmha_launch(bool diff, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const FmhaArgs& a, long long num_ctas,
                        cudaStream_t stream) {
  if (diff) return bf16 ? launch_masked<true, true>(tq, tk, tv, a, num_ctas, stream)
                        : launch_masked<true, false>(tq, tk, tv, a, num_ctas, stream);
  return bf16 ? launch_masked<false, true>(tq, tk, tv, a, num_ctas, stream)
              : launch_masked<false, false>(tq, tk, tv, a, num_ctas, stream);
}

}  // namespace sa
