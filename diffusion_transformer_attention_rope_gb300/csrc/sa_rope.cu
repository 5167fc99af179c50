// sa_rope.cu -- RoPE pre-pass: q' = RoPE(q), k' = RoPE(k) in FP32, cast back to fp16/bf16.
//
// HF discussion #3 "fp16mixed attention-core fix", section "The bug": apply_rotary_pos_emb
// computes in FP32 and finishes with a cast to the output dtype, so attention then runs on
// fp16/bf16 q, k.
// Rotate-half over the full head dim (d = 64): pair (i, i + 32) at position p turns by
// theta = p * inv_freq[i], inv_freq[i] = base^(-2i/64) held as FP32.  The angle itself is an
// FP32 product and sin/cos are the full-precision single-precision functions: the sa3_trt
// README ("Retired: bf16") shows what a low-precision angle does at long sequence lengths.
//
// With a table pointer the pass also writes each position's 32 (cos, sin) pairs (FP32), which
// the attention kernel uses to rotate q in its prologue; q is then not touched here.
//
// Optional QK-RMSNorm (the pages run RMSNorm and RoPE next to attention in FP32, so that
// variances cannot overflow fp16): each row is first scaled by gamma / sqrt(mean(x^2) + eps) in FP32,
// then rotated, then cast once.  The 4 threads of a row (consecutive lanes) add their partial
// sums of squares with a 2-step butterfly.
//
// One block rotates 32 positions of every plane in its slice of planes (a plane is one
// (batch, head, map) sequence of L rows).  A thread owns 8 rotation pairs of one position
// (two 16-byte chunks per row) and up to kPlaneBatch planes at a time: it issues all the loads
// of a batch first, then computes its 8 (cos, sin) pairs once, then rotates and stores, so
// many bytes are in flight per thread.  The pass is HBM-bound: q, k read once, q', k' written
// once.  Each block signals early that the dependent attention launch may start (its CTAs
// then only prepare; they wait for this grid before reading q', k').
//
// Two more forms: the k pass as a few 512-thread blocks walking the same items (for a call
// whose attention grid leaves SMs idle: the pass then stays on those SMs), and the (cos, sin)
// table alone (the handle's table of positions 0 .. capacity - 1), both with the same
// per-element arithmetic.
#include "sa_kernels.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kRopeRows = 32;      // positions per block
constexpr int kRopeThreads = 128;  // 32 positions x 4 groups of 8 rotation pairs
constexpr int kPlaneBatch = 4;     // planes whose loads are issued together

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(uint16_t* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The row's inverse RMS from this thread's partial sum of squares (lanes of a row: gmask).
__device__ __forceinline__ float row_inv_rms(float t, unsigned gmask, float eps) {
  const float u = t + __shfl_xor_sync(gmask, t, 1);
  return qknorm_inv_rms(u + __shfl_xor_sync(gmask, u, 2), eps);
}

// The gammas in shared memory (q then k; registers are what limits this pass's occupancy); a
// thread reads those of its 16 values, [8g, 8g + 8) and [32 + 8g, 32 + 8g + 8).
template <bool NORM, int THREADS>
__device__ __forceinline__ void load_gamma(const RopeArgs& a, float (*s_gamma)[kHeadDim]) {
  if (NORM) {
    for (int i = threadIdx.x; i < 2 * kHeadDim; i += THREADS)
      s_gamma[i / kHeadDim][i % kHeadDim] = i < kHeadDim ? a.gamma_q[i] : a.gamma_k[i - kHeadDim];
    __syncthreads();
  }
}

// One item of the pass: positions [bx ROWS, (bx + 1) ROWS) of the planes of slice `by`
// (planes_per_block planes), four threads per position.
// WITH_Q: rotate q as well as k (false when the attention kernel rotates q in its prologue).
// NORM: QK-RMSNorm of every row before its rotation.
template <bool BF16, bool WITH_Q, bool NORM, int ROWS>
__device__ __forceinline__ void rope_item(const RopeArgs& a, const float (*s_gamma)[kHeadDim], int bx,
                                          long long by) {
  const int r = threadIdx.x >> 2;  // position within the item
  const int g = threadIdx.x & 3;   // group of 8 pairs: pairs [8g, 8g + 8)
  const int l = bx * ROWS + r;
  if (l >= a.L) return;            // (all 4 lanes of a row leave together)
  const unsigned gmask = 0xFu << (threadIdx.x & 28);
  const long long first = by * a.planes_per_block;
  long long last = first + a.planes_per_block;
  if (last > a.planes) last = a.planes;
  const size_t row_stride = static_cast<size_t>(a.L) * kHeadDim;
  const size_t base = static_cast<size_t>(l) * kHeadDim + 8 * g;

  float c[8], s[8];
  bool have_cs = false;
  for (long long p0 = first; p0 < last; p0 += kPlaneBatch) {
    const int n = static_cast<int>(last - p0 < kPlaneBatch ? last - p0 : kPlaneBatch);
    uint4 qlo[kPlaneBatch], qhi[kPlaneBatch], klo[kPlaneBatch], khi[kPlaneBatch];
#pragma unroll
    for (int i = 0; i < kPlaneBatch; ++i) {
      if (i < n) {
        const size_t off = static_cast<size_t>(p0 + i) * row_stride + base;
        if (WITH_Q) {
          qlo[i] = ld_stream(a.q + off);
          qhi[i] = ld_stream(a.q + off + 32);
        }
        klo[i] = ld_stream(a.k + off);
        khi[i] = ld_stream(a.k + off + 32);
      }
    }
    if (!have_cs) {
      const int p = a.positions ? a.positions[l] : l;
      const float pf = static_cast<float>(p);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float theta = __fmul_rn(pf, a.inv_freq[8 * g + i]);
        sincosf(theta, &s[i], &c[i]);
      }
      have_cs = true;
      if (a.cs != nullptr && by == 0) {
        // this position's pairs [8g, 8g + 8) of the (cos, sin) table for the Q prologue; the
        // table is [16][L] float4 (cos_2m, cos_2m+1, sin_2m, sin_2m+1 of position l at [m][l]), so
        // that the prologue's loads of consecutive rows are contiguous and each (cos, cos) and
        // (sin, sin) pair is one 64-bit operand of the paired FP32 rotation
        float4* t = reinterpret_cast<float4*>(a.cs);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          t[static_cast<size_t>(4 * g + i) * a.L + l] = make_float4(c[2 * i], c[2 * i + 1], s[2 * i], s[2 * i + 1]);
      }
    }
#pragma unroll
    for (int i = 0; i < kPlaneBatch; ++i) {
      if (i < n) {
        const size_t off = static_cast<size_t>(p0 + i) * row_stride + base;
        uint4 lo, hi;
        if (NORM) {
          float sl[8], sh[8];
          if (WITH_Q) {
            const float inv = row_inv_rms(sumsq8<BF16>(qlo[i]) + sumsq8<BF16>(qhi[i]), gmask, a.eps);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              sl[j] = __fmul_rn(inv, s_gamma[0][8 * g + j]);
              sh[j] = __fmul_rn(inv, s_gamma[0][32 + 8 * g + j]);
            }
            rope_rotate8_scaled<BF16>(qlo[i], qhi[i], c, s, sl, sh, lo, hi);
            st_v4(a.q_out + off, lo);
            st_v4(a.q_out + off + 32, hi);
          }
          const float inv = row_inv_rms(sumsq8<BF16>(klo[i]) + sumsq8<BF16>(khi[i]), gmask, a.eps);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            sl[j] = __fmul_rn(inv, s_gamma[1][8 * g + j]);
            sh[j] = __fmul_rn(inv, s_gamma[1][32 + 8 * g + j]);
          }
          rope_rotate8_scaled<BF16>(klo[i], khi[i], c, s, sl, sh, lo, hi);
        } else {
          if (WITH_Q) {
            rope_rotate8<BF16>(qlo[i], qhi[i], c, s, lo, hi);
            st_v4(a.q_out + off, lo);
            st_v4(a.q_out + off + 32, hi);
          }
          rope_rotate8<BF16>(klo[i], khi[i], c, s, lo, hi);
        }
        st_v4(a.k_out + off, lo);
        st_v4(a.k_out + off + 32, hi);
      }
    }
  }
}

template <bool BF16, bool WITH_Q, bool NORM>
__device__ __forceinline__ void rope_body(const RopeArgs& a) {
  // Let the dependent attention grid begin its prologue while this grid streams.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float s_gamma[2][kHeadDim];
  load_gamma<NORM, kRopeThreads>(a, s_gamma);
  rope_item<BF16, WITH_Q, NORM, kRopeRows>(a, s_gamma, blockIdx.x, blockIdx.y);
}

template <bool BF16, bool WITH_Q>
__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const __grid_constant__ RopeArgs a) {
  rope_body<BF16, WITH_Q, false>(a);
}

template <bool BF16, bool WITH_Q>
__global__ void __launch_bounds__(kRopeThreads) rope_norm_kernel(const __grid_constant__ RopeArgs a) {
  rope_body<BF16, WITH_Q, true>(a);
}

// The k-only pass walking its items with a grid of at most the SMs the attention grid leaves
// idle (items: kSideRows positions of planes_per_block planes).
constexpr int kSideRows = kRopeSideThreads / 4;

template <bool BF16, bool NORM>
__global__ void __launch_bounds__(kRopeSideThreads) rope_side_kernel(const __grid_constant__ RopeArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float s_gamma[2][kHeadDim];
  load_gamma<NORM, kRopeSideThreads>(a, s_gamma);
  const int nx = (a.L + kSideRows - 1) / kSideRows;
  const long long items = static_cast<long long>(nx) * ((a.planes + a.planes_per_block - 1) / a.planes_per_block);
  for (long long item = blockIdx.x; item < items; item += gridDim.x)
    rope_item<BF16, false, NORM, kSideRows>(a, s_gamma, static_cast<int>(item % nx), item / nx);
}

// The (cos, sin) table alone, for positions 0 .. L - 1 (or a.positions): four threads per
// position, 8 pairs each, with the arithmetic of the pass above (so the table has its bits).
__global__ void __launch_bounds__(kRopeThreads) rope_table_kernel(const __grid_constant__ RopeArgs a) {
  const int r = threadIdx.x >> 2, g = threadIdx.x & 3;
  const int l = blockIdx.x * kRopeRows + r;
  if (l >= a.L) return;
  const float pf = static_cast<float>(a.positions ? a.positions[l] : l);
  float c[8], s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sincosf(__fmul_rn(pf, a.inv_freq[8 * g + i]), &s[i], &c[i]);
  float4* t = reinterpret_cast<float4*>(a.cs);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    t[static_cast<size_t>(4 * g + i) * a.L + l] = make_float4(c[2 * i], c[2 * i + 1], s[2 * i], s[2 * i + 1]);
}

// Resident blocks per SM of one variant (the fewer of its fp16 and bf16 forms).
template <bool WITH_Q, bool NORM>
int blocks_per_sm() {
  const void* fns[2] = {
      NORM ? reinterpret_cast<const void*>(rope_norm_kernel<false, WITH_Q>) : reinterpret_cast<const void*>(rope_kernel<false, WITH_Q>),
      NORM ? reinterpret_cast<const void*>(rope_norm_kernel<true, WITH_Q>) : reinterpret_cast<const void*>(rope_kernel<true, WITH_Q>)};
  int least = 1 << 30;
  for (const void* f : fns) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kRopeThreads, 0) != cudaSuccess) return 1;
    least = n < least ? n : least;
  }
  return least > 0 ? least : 1;
}

template <bool BF16, bool WITH_Q>
void launch_variant(const RopeArgs& a, dim3 grid, cudaStream_t stream) {
  if (a.qk_norm) rope_norm_kernel<BF16, WITH_Q><<<grid, kRopeThreads, 0, stream>>>(a);
  else rope_kernel<BF16, WITH_Q><<<grid, kRopeThreads, 0, stream>>>(a);
}

}  // namespace

int rope_blocks_per_sm(bool with_q, bool qk_norm) {
  if (with_q) return qk_norm ? blocks_per_sm<true, true>() : blocks_per_sm<true, false>();
  return qk_norm ? blocks_per_sm<false, true>() : blocks_per_sm<false, false>();
}

cudaError_t rope_launch(const RopeArgs& a_in, bool bf16, int num_sms, int blocks_per_sm,
                        cudaStream_t stream) {
  RopeArgs a = a_in;
  const long long bx = (a.L + kRopeRows - 1) / kRopeRows;
  // A thread issues the loads of up to kPlaneBatch planes at once.  Take the fewest planes per
  // block (the (cos, sin) pairs are computed once per thread and reused for its planes) that
  // fits the grid into what is resident at once, up to one batch per thread; past that, more
  // blocks (waves) rather than more serial batches per thread.
  const long long resident = static_cast<long long>(num_sms > 0 ? num_sms : 148) *
                             (blocks_per_sm > 0 ? blocks_per_sm : 1);
  long long ppb = 1;
  while (ppb < a.planes && ppb < kPlaneBatch && bx * ((a.planes + ppb - 1) / ppb) > resident) ++ppb;
  long long by = (a.planes + ppb - 1) / ppb;
  if (by > 65535) {
    by = 65535;
    ppb = (a.planes + by - 1) / by;
    by = (a.planes + ppb - 1) / ppb;
  }
  a.planes_per_block = static_cast<int>(ppb);
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(by));
  const bool with_q = a.q != nullptr;
  if (bf16) {
    if (with_q) launch_variant<true, true>(a, grid, stream);
    else launch_variant<true, false>(a, grid, stream);
  } else {
    if (with_q) launch_variant<false, true>(a, grid, stream);
    else launch_variant<false, false>(a, grid, stream);
  }
  return cudaGetLastError();
}

cudaError_t rope_side_launch(const RopeArgs& a_in, bool bf16, int blocks, cudaStream_t stream) {
  RopeArgs a = a_in;
  a.q = nullptr;
  a.q_out = nullptr;
  a.cs = nullptr;
  a.planes_per_block = static_cast<int>(a.planes < kPlaneBatch ? a.planes : kPlaneBatch);
  const int nx = (a.L + kSideRows - 1) / kSideRows;
  const long long items = static_cast<long long>(nx) * ((a.planes + a.planes_per_block - 1) / a.planes_per_block);
  const unsigned grid = static_cast<unsigned>(items < blocks ? items : blocks);
  if (bf16) {
    if (a.qk_norm) rope_side_kernel<true, true><<<grid, kRopeSideThreads, 0, stream>>>(a);
    else rope_side_kernel<true, false><<<grid, kRopeSideThreads, 0, stream>>>(a);
  } else {
    if (a.qk_norm) rope_side_kernel<false, true><<<grid, kRopeSideThreads, 0, stream>>>(a);
    else rope_side_kernel<false, false><<<grid, kRopeSideThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t rope_table_launch(const RopeArgs& a, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((a.L + kRopeRows - 1) / kRopeRows);
  rope_table_kernel<<<grid, kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
