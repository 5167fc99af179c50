// sa_api.cu -- the C ABI declared in include/sa_attn.h: host-side argument checks, the
// per-device handle, TMA descriptor encoding and the two launches (RoPE pre-pass, attention).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "sa_attn.h"
#include "sa_kernels.h"

struct sa_attn_s {
  int device;
  int num_sms;
  int rope_blocks_per_sm[2][2];   // RoPE pass: [rotates q too][QK-RMSNorm]
  float rope_base;
  float inv_freq[sa::kHeadDim / 2];
  int* d_err;  // 4-byte device error word
  // (cos, sin) table of positions 0 .. cs_cap - 1 ([16][cs_cap] float4), written once at
  // creation: calls with the default positions and L <= cs_cap read it instead of a per-call
  // table (nullptr / 0 if it could not be allocated)
  float2* d_cs;
  int cs_cap;
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  unsigned long long timeout_ns;
  // sa_rope_attn_host: copy-in, copy-out and per-chunk compute streams, and their events
  cudaStream_t hs_in, hs_out, hs_comp[sa::kHostChunks];
  cudaEvent_t he_entry, he_in[sa::kHostChunks], he_done[sa::kHostChunks], he_exit;
  bool host_ready;
  // sa_rope_attn_noalloc: device address of the library's static scratch array in this
  // handle's context, looked up on the handle's first call of that function (nullptr before)
  void* noalloc_scratch;
};

namespace {

thread_local char g_msg[512] = "";

sa_status fail(sa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

sa_status ok() {
  g_msg[0] = '\0';
  return SA_OK;
}

// Switches to `dev` for the lifetime of the object and restores the caller's device.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// 3-D tiled map over a [planes][rows][cols] array of 2-byte elements: box = 64 cols x box_rows
// rows x 1 plane, 128-byte swizzle (the layout the tcgen05 descriptors expect).  Rows past the
// end of a plane read as zeros.
bool encode_map(const sa_attn_s* h, CUtensorMap* m, const void* base, bool bf16, uint64_t cols,
                uint64_t rows, uint64_t planes, uint32_t box_rows = sa::kBlockN) {
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {cols * 2, cols * 2 * rows};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = h->encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The FP32 form: [planes][rows][cols] FP32 (rows row_pitch elements apart, cols if 0), box = 32
// cols (128 bytes) x box_rows x 1 plane, 128-byte swizzle, elements past the end read as zeros.
bool encode_map_f32(const sa_attn_s* h, CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                    uint64_t planes, uint32_t box_rows, uint64_t row_pitch = 0) {
  const uint64_t pitch = row_pitch ? row_pitch : cols;   // elements per row in memory
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {pitch * 4, pitch * 4 * rows};
  const cuuint32_t box[3] = {32, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = h->encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Entry points whose 16-bit-only forms (the Q prologue, the QK-RMSNorm, host buffers) have no
// FP32 counterpart.
sa_status reject_fp32(const char* fn, sa_dtype dtype) {
  if (dtype == SA_FP32)
    return fail(SA_ERR_UNSUPPORTED, "%s: SA_FP32 is supported by sa_rope_attn, sa_rope_attn_noalloc, "
                "sa_rope_qk and sa_attn_fwd only", fn);
  return SA_OK;
}

bool qk_elems(int B, int H, int L, int nmaps, size_t* out) {
  if (B <= 0 || H <= 0 || L <= 0) return false;
  const unsigned long long n = static_cast<unsigned long long>(B) * H * nmaps * L * sa::kHeadDim;
  if (n >= (1ull << 40)) return false;
  *out = static_cast<size_t>(n);
  return true;
}


// Streams and events of sa_rope_attn_host, created with the handle (false if any failed; the
// host entry then reports SA_ERR_CUDA).
bool create_host_streams(sa_attn_s* h) {
  bool good = cudaStreamCreateWithFlags(&h->hs_in, cudaStreamNonBlocking) == cudaSuccess;
  good = good && cudaStreamCreateWithFlags(&h->hs_out, cudaStreamNonBlocking) == cudaSuccess;
  for (int c = 0; c < sa::kHostChunks; ++c) {
    good = good && cudaStreamCreateWithFlags(&h->hs_comp[c], cudaStreamNonBlocking) == cudaSuccess;
    good = good && cudaEventCreateWithFlags(&h->he_in[c], cudaEventDisableTiming) == cudaSuccess;
    good = good && cudaEventCreateWithFlags(&h->he_done[c], cudaEventDisableTiming) == cudaSuccess;
  }
  good = good && cudaEventCreateWithFlags(&h->he_entry, cudaEventDisableTiming) == cudaSuccess;
  good = good && cudaEventCreateWithFlags(&h->he_exit, cudaEventDisableTiming) == cudaSuccess;
  return good;
}

// Positions the handle's (cos, sin) table covers (4 MiB of device memory).
constexpr int kTableCap = 16384;

// The handle's table of positions 0 .. kTableCap - 1, written once here with the RoPE pass's
// arithmetic.  Without it (allocation failed) every call computes its own table.
void create_table(sa_attn_s* h) {
  h->d_cs = nullptr;
  h->cs_cap = 0;
  void* p = nullptr;
  if (cudaMalloc(&p, static_cast<size_t>(kTableCap) * (sa::kHeadDim / 2) * sizeof(float2)) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  sa::RopeArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.cs = static_cast<float2*>(p);
  ra.L = kTableCap;
  std::memcpy(ra.inv_freq, h->inv_freq, sizeof(ra.inv_freq));
  if (sa::rope_table_launch(ra, nullptr) != cudaSuccess || cudaStreamSynchronize(nullptr) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p);
    return;
  }
  h->d_cs = static_cast<float2*>(p);
  h->cs_cap = kTableCap;
}

// Releases the handle's streams, events and table.
void destroy_host_streams(sa_attn_s* h) {
  if (h->d_cs) cudaFree(h->d_cs);
  h->d_cs = nullptr;
  // (destroying a null stream or event handle is harmless)
  if (h->hs_in) cudaStreamDestroy(h->hs_in);
  if (h->hs_out) cudaStreamDestroy(h->hs_out);
  for (int c = 0; c < sa::kHostChunks; ++c) {
    if (h->hs_comp[c]) cudaStreamDestroy(h->hs_comp[c]);
    if (h->he_in[c]) cudaEventDestroy(h->he_in[c]);
    if (h->he_done[c]) cudaEventDestroy(h->he_done[c]);
  }
  if (h->he_entry) cudaEventDestroy(h->he_entry);
  if (h->he_exit) cudaEventDestroy(h->he_exit);
}

// Shape / dtype checks shared by the entry points.
sa_status check_shape(const char* fn, int B, int H, int L, int d, sa_dtype dtype, bool diff) {
  if (B <= 0 || H <= 0 || L <= 0)
    return fail(SA_ERR_INVALID_ARG, "%s: B, H, L must be >= 1 (got %d, %d, %d)", fn, B, H, L);
  if (L >= sa::kMaxL)
    return fail(SA_ERR_UNSUPPORTED, "%s: L = %d exceeds the supported maximum %d", fn, L, sa::kMaxL - 1);
  if (d != sa::kHeadDim)
    return fail(SA_ERR_UNSUPPORTED, "%s: head dim d = %d; only d = 64 is supported", fn, d);
  if (dtype != SA_FP16 && dtype != SA_BF16 && dtype != SA_FP32)
    return fail(SA_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, static_cast<int>(dtype));
  if (dtype == SA_FP32 && !diff)
    return fail(SA_ERR_UNSUPPORTED, "%s: SA_FP32 inputs are supported for differential attention "
                "(lambda != NULL, two maps) only", fn);
  if (diff && H > sa::kMaxDiffHeads)
    return fail(SA_ERR_UNSUPPORTED, "%s: differential attention supports H <= %d (got %d)", fn,
                sa::kMaxDiffHeads, H);
  size_t n = 0;
  const int dv = diff ? 2 * d : d;
  if (!qk_elems(B, H, L, diff ? 2 : 1, &n) ||
      static_cast<unsigned long long>(B) * H * L * dv >= (1ull << 40))
    return fail(SA_ERR_INVALID_ARG, "%s: tensor sizes overflow", fn);
  const int rows = sa::fmha_rows_per_cta(diff);
  if (static_cast<long long>(B) * H * ((L + rows - 1) / rows) >= (1ll << 31))
    return fail(SA_ERR_UNSUPPORTED, "%s: too many query tiles for one launch", fn);
  return SA_OK;
}

sa_status check_lambda(const char* fn, const float* lambda, int H) {
  if (!lambda) return SA_OK;
  for (int i = 0; i < H; ++i)
    if (!std::isfinite(lambda[i]))
      return fail(SA_ERR_INVALID_ARG, "%s: lambda[%d] is not finite", fn, i);
  return SA_OK;
}

// QK-RMSNorm parameters as the kernels take them (gamma NULL: all ones).
struct QkNorm {
  float eps;
  float gamma_q[sa::kHeadDim];
  float gamma_k[sa::kHeadDim];
};

sa_status make_qknorm(const char* fn, const float* gamma_q, const float* gamma_k, float eps, QkNorm* n) {
  if (!std::isfinite(eps) || eps < 0.0f)
    return fail(SA_ERR_INVALID_ARG, "%s: eps must be finite and >= 0 (got %g)", fn, static_cast<double>(eps));
  n->eps = eps;
  for (int i = 0; i < sa::kHeadDim; ++i) {
    n->gamma_q[i] = gamma_q ? gamma_q[i] : 1.0f;
    n->gamma_k[i] = gamma_k ? gamma_k[i] : 1.0f;
    if (!std::isfinite(n->gamma_q[i]) || !std::isfinite(n->gamma_k[i]))
      return fail(SA_ERR_INVALID_ARG, "%s: gamma_q[%d] or gamma_k[%d] is not finite", fn, i, i);
  }
  return SA_OK;
}

// q == nullptr: rotate k only and write the (cos, sin) table cs (for the Q prologue).
// nrm: QK-RMSNorm before the rotation, or nullptr.
// side_blocks > 0 (q == nullptr, cs == nullptr): the k pass as at most that many blocks, on SMs
// the attention grid leaves idle.
sa_status launch_rope(const sa_attn_s* h, const void* q, const void* k, const int32_t* positions,
                      void* q_rot, void* k_rot, int B, int H, int L, int nmaps, sa_dtype dtype,
                      sa_stream_t stream, void* cs = nullptr, const QkNorm* nrm = nullptr,
                      int side_blocks = 0) {
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);
  sa::RopeArgs ra;
  ra.q = static_cast<const uint16_t*>(q);
  ra.k = static_cast<const uint16_t*>(k);
  ra.q_out = static_cast<uint16_t*>(q_rot);
  ra.k_out = static_cast<uint16_t*>(k_rot);
  ra.cs = static_cast<float2*>(cs);
  ra.positions = positions;
  ra.planes = static_cast<long long>(B) * H * nmaps;
  ra.L = L;
  ra.planes_per_block = 1;
  std::memcpy(ra.inv_freq, h->inv_freq, sizeof(ra.inv_freq));
  ra.qk_norm = nrm != nullptr;
  ra.eps = nrm ? nrm->eps : 0.0f;
  for (int i = 0; i < sa::kHeadDim; ++i) {
    ra.gamma_q[i] = nrm ? nrm->gamma_q[i] : 1.0f;
    ra.gamma_k[i] = nrm ? nrm->gamma_k[i] : 1.0f;
  }
  cudaError_t e = side_blocks > 0
      ? sa::rope_side_launch(ra, dtype == SA_BF16, side_blocks, reinterpret_cast<cudaStream_t>(stream))
      : sa::rope_launch(ra, dtype == SA_BF16, h->num_sms, h->rope_blocks_per_sm[q != nullptr][nrm != nullptr],
                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "RoPE launch: %s", cudaGetErrorString(e));
  return ok();
}

// Key tiles visited by query block qb (the kernel's own rule).
int block_tiles_host(int L, int window, int rows, int qb) {
  if (window < 0) return (L - 1) / sa::kBlockN + 1;
  const int q0 = qb * rows;
  const int q_last = std::min(L, q0 + rows) - 1;
  const int first = std::max(0, q0 - window);
  return (std::min(L - 1, q_last + window) - first) / sa::kBlockN + 1;
}

// Every launch gets its own epoch: it tags the unit counters of the split region, so they
// never need clearing by the caller.
std::atomic<unsigned> g_epoch{0};

// Bytes of the split region for this shape: one 8-byte counter per unit, then one partial-result
// slot per piece CTA (at most kMaxPieces).
size_t split_bytes(int B, int H, int L, bool diff) {
  const int rows = sa::fmha_rows_per_cta(diff);
  const unsigned long long units = static_cast<unsigned long long>(B) * H * ((L + rows - 1) / rows);
  return align256(units * 8) +
         align256(static_cast<size_t>(sa::kMaxPieces) * sa::fmha_partial_floats(diff) * sizeof(float));
}

// The attention launch's grid: one CTA per unit, except that when the units leave the GPU's
// last wave partly empty and a split region is given, the tail units (those of that last wave)
// are cut into tail_k pieces of their key range, one CTA each, with tail_k as large as the wave
// allows.
struct AttnGrid {
  long long units, ctas;
  int n_qblocks, window, whole_ctas, tail_k;
};

AttnGrid attn_grid(const sa_attn_s* h, int B, int H, int L, int window, bool diff, bool split) {
  AttnGrid g;
  const int rows = sa::fmha_rows_per_cta(diff);
  g.n_qblocks = (L + rows - 1) / rows;
  g.window = (window < 0 || window >= L - 1) ? -1 : window;
  g.units = static_cast<long long>(B) * H * g.n_qblocks;
  g.whole_ctas = static_cast<int>(g.units);
  g.tail_k = 1;
  g.ctas = g.units;
  const long long G = std::min<long long>(h->num_sms, sa::kMaxPieces);
  const long long tail = g.units % G;
  if (split && tail > 0) {
    int min_nt = 1 << 30;
    for (int qb = 0; qb < g.n_qblocks; ++qb) min_nt = std::min(min_nt, block_tiles_host(L, g.window, rows, qb));
    const long long k = std::min<long long>(std::min<long long>(G / tail, min_nt), sa::kMaxTailK);
    if (k >= 2) {
      g.whole_ctas = static_cast<int>(g.units - tail);
      g.tail_k = static_cast<int>(k);
      g.ctas = (g.units - tail) + tail * k;
    }
  }
  return g;
}

// SMs an attention grid of `ctas` CTAs (one per SM) leaves idle, if the k pass should run on
// them (0: it runs on every SM, before the attention CTAs can start).  The attention CTAs then
// start with the pass and do their setup and Q prologue meanwhile; only their K loads wait
// for it.  Taken when the pass stays short there: at least 8 idle SMs and at most 256 KiB of
// k for each.
int side_sms(const sa_attn_s* h, long long ctas, long long k_bytes) {
  const long long idle = h->num_sms - ctas;
  if (idle < 8 || k_bytes > idle * 256 * 1024) return 0;
  return static_cast<int>(idle);
}

// Differential attention with a window of at most kSwaMaxWindow: the narrow-window kernel, one
// CTA per SM walking runs of query blocks (q rotated in its prologue with the table cs, or q'
// rotated already when cs is nullptr).
sa_status launch_attn_swa(const sa_attn_s* h, const void* q, const void* k_rot, const void* v, void* out, int B,
                          int H, int L, int window, const float* lambda, bool bf16, sa_stream_t stream,
                          const void* cs, int cs_stride, bool cs_static, const QkNorm* nrm) {
  const unsigned long long planes_qk = static_cast<unsigned long long>(B) * H * 2;
  const unsigned long long planes_v = static_cast<unsigned long long>(B) * H;
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  if (!aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (!encode_map(h, &tm_q, q, bf16, sa::kHeadDim, L, planes_qk, sa::kBlockM) ||
      !encode_map(h, &tm_k, k_rot, bf16, sa::kHeadDim, L, planes_qk, 64) ||
      !encode_map(h, &tm_v, v, bf16, 2 * sa::kHeadDim, L, planes_v, 64) ||
      !encode_map(h, &tm_o, out, bf16, 2 * sa::kHeadDim, L, planes_v, 32))
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor map");
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);
  sa::FmhaSwaArgs fa;
  std::memset(&fa, 0, sizeof(fa));
  fa.out = out;
  fa.err = h->d_err;
  fa.L = L;
  fa.H = H;
  fa.n_qblocks = (L + sa::kBlockM - 1) / sa::kBlockM;
  fa.window = window;
  fa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(sa::kHeadDim)));
  fa.timeout_ns = h->timeout_ns;
  fa.units = static_cast<long long>(B) * H * fa.n_qblocks;
  fa.cs = static_cast<const float2*>(cs);
  fa.cs_stride = cs_stride > 0 ? cs_stride : L;
  fa.cs_static = cs_static;
  for (int i = 0; i < H; ++i) fa.lambda[i] = lambda[i];
  fa.qk_norm = nrm != nullptr;   // (with cs: the prologue normalises each raw q row)
  fa.eps = nrm ? nrm->eps : 0.0f;
  for (int i = 0; i < sa::kHeadDim; ++i) fa.gamma_q[i] = nrm ? nrm->gamma_q[i] : 1.0f;
  const int ctas = static_cast<int>(std::min<long long>(fa.units, h->num_sms));
  const cudaError_t e =
      sa::fmha_swa_launch(bf16, tm_q, tm_k, tm_v, tm_o, fa, ctas, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "attention (narrow window) launch: %s", cudaGetErrorString(e));
  return ok();
}

// cs == nullptr: q_rot is rotated already; else q_rot is the raw q and the kernel rotates it
// in its prologue with the (cos, sin) table cs (row stride cs_stride, L if 0; cs_static: the
// handle's table, which no kernel of this call writes).
sa_status launch_attn(const sa_attn_s* h, const void* q_rot, const void* k_rot, const void* v,
                      void* out, int B, int H, int L, int window, const float* lambda,
                      sa_dtype dtype, void* split_ws, sa_stream_t stream, const void* cs = nullptr,
                      const QkNorm* nrm = nullptr, int cs_stride = 0, bool cs_static = false) {
  const bool diff = lambda != nullptr;
  const bool bf16 = dtype == SA_BF16;
  const int d = sa::kHeadDim;
  const int dv = diff ? 2 * d : d;
  const unsigned long long planes_qk = static_cast<unsigned long long>(B) * H * (diff ? 2 : 1);
  const unsigned long long planes_v = static_cast<unsigned long long>(B) * H;
  const int wnd = (window < 0 || window >= L - 1) ? -1 : window;
  if (diff && wnd >= 0 && wnd <= sa::kSwaMaxWindow)
    return launch_attn_swa(h, q_rot, k_rot, v, out, B, H, L, wnd, lambda, bf16, stream, cs, cs_stride, cs_static,
                           nrm);
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_map(h, &tm_q, q_rot, bf16, d, L, planes_qk) ||
      !encode_map(h, &tm_k, k_rot, bf16, d, L, planes_qk) ||
      !encode_map(h, &tm_v, v, bf16, dv, L, planes_v))
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor map");
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);
  sa::FmhaArgs fa;
  std::memset(&fa, 0, sizeof(fa));
  fa.out = out;
  fa.err = h->d_err;
  fa.L = L;
  fa.H = H;
  const AttnGrid g = attn_grid(h, B, H, L, window, diff, split_ws != nullptr);
  fa.n_qblocks = g.n_qblocks;
  fa.window = g.window;
  fa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  fa.timeout_ns = h->timeout_ns;
  fa.cs = static_cast<const float2*>(cs);
  fa.cs_stride = cs_stride > 0 ? cs_stride : L;
  fa.cs_static = cs_static;
  fa.qk_norm = nrm != nullptr;   // (with cs: the Q prologue normalises each raw q row)
  fa.eps = nrm ? nrm->eps : 0.0f;
  for (int i = 0; i < sa::kHeadDim; ++i) fa.gamma_q[i] = nrm ? nrm->gamma_q[i] : 1.0f;
  if (diff)
    for (int i = 0; i < H; ++i) fa.lambda[i] = lambda[i];
  fa.whole_ctas = g.whole_ctas;
  fa.tail_k = g.tail_k;
  const long long ctas = g.ctas;
  if (g.tail_k > 1) {
    uint8_t* ws = static_cast<uint8_t*>(split_ws);
    fa.counters = reinterpret_cast<unsigned long long*>(ws);
    fa.partials = reinterpret_cast<float*>(ws + align256(static_cast<size_t>(g.units) * 8));
    unsigned ep = g_epoch.fetch_add(1u) + 1u;
    if (ep == 0) ep = g_epoch.fetch_add(1u) + 1u;
    fa.epoch = ep;
  }
  fa.wave = h->num_sms;
  cudaError_t e = sa::fmha_launch(diff, bf16, tm_q, tm_k, tm_v, fa, ctas, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return ok();
}

// Keys per row of the FP32 form's v^T (rows of 16 bytes for its tensor map).
int f32_lpad(int L) { return (L + 3) & ~3; }

size_t f32_vt_bytes(int B, int H, int L) {
  return align256(static_cast<size_t>(B) * H * 2 * sa::kHeadDim * f32_lpad(L) * 4);
}

// The FP32 form's pre-pass: q' and k' (both maps) rotated in FP32 and rounded to TF32 (q == nullptr:
// none), and v^T [B*H][128][L_pad] rounded to TF32 (v == nullptr: none).
sa_status launch_rope_f32(const sa_attn_s* h, const void* q, const void* k, const int32_t* positions,
                          void* q_rot, void* k_rot, int B, int H, int L, sa_stream_t stream,
                          const void* v = nullptr, void* v_t = nullptr) {
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);
  sa::RopeF32Args ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.q = static_cast<const float*>(q);
  ra.k = static_cast<const float*>(k);
  ra.q_out = static_cast<float*>(q_rot);
  ra.k_out = static_cast<float*>(k_rot);
  ra.positions = positions;
  ra.planes = static_cast<long long>(B) * H * 2;
  ra.L = L;
  std::memcpy(ra.inv_freq, h->inv_freq, sizeof(ra.inv_freq));
  ra.v = static_cast<const float*>(v);
  ra.v_t = static_cast<float*>(v_t);
  ra.planes_v = static_cast<long long>(B) * H;
  ra.L_pad = f32_lpad(L);
  const cudaError_t e = sa::rope_f32_launch(ra, h->num_sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "RoPE (FP32) launch: %s", cudaGetErrorString(e));
  return ok();
}

// The FP32 form's attention stage on q', k' and v^T (TF32 products), one CTA per 128-row query
// block.
sa_status launch_attn_f32(const sa_attn_s* h, const void* q_rot, const void* k_rot, const void* v_t, void* out,
                          int B, int H, int L, int window, const float* lambda, sa_stream_t stream) {
  const int d = sa::kHeadDim;
  const unsigned long long planes_qk = static_cast<unsigned long long>(B) * H * 2;
  const unsigned long long planes_v = static_cast<unsigned long long>(B) * H;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_map_f32(h, &tm_q, q_rot, d, L, planes_qk, sa::kBlockM) ||
      !encode_map_f32(h, &tm_k, k_rot, d, L, planes_qk, 64) ||
      !encode_map_f32(h, &tm_v, v_t, L, 2 * d, planes_v, sa::kBlockM, f32_lpad(L)))
    return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor map");
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);
  sa::FmhaF32Args fa;
  std::memset(&fa, 0, sizeof(fa));
  fa.out = static_cast<float*>(out);
  fa.err = h->d_err;
  fa.L = L;
  fa.H = H;
  fa.n_qblocks = (L + sa::kBlockM - 1) / sa::kBlockM;
  fa.window = (window < 0 || window >= L - 1) ? -1 : window;
  fa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  fa.timeout_ns = h->timeout_ns;
  for (int i = 0; i < H; ++i) fa.lambda[i] = lambda[i];
  const long long ctas = static_cast<long long>(B) * H * fa.n_qblocks;
  const cudaError_t e = sa::fmha_tf32_launch(tm_q, tm_k, tm_v, fa, ctas, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "attention (TF32) launch: %s", cudaGetErrorString(e));
  return ok();
}

// sa_rope_attn's FP32 workspace: q', k', v^T.
size_t f32_ws_bytes(int B, int H, int L) {
  size_t n = 0;
  if (!qk_elems(B, H, L, 2, &n)) return 0;
  return 2 * align256(n * 4) + f32_vt_bytes(B, H, L);
}

}  // namespace

namespace sa {

// Library-internal hooks used by sa_noalloc.cu (not exported).
sa_status set_error(sa_status st, const char* msg) { return fail(st, "%s", msg); }

int handle_device(sa_attn_t h) { return h->device; }

void** handle_noalloc_slot(sa_attn_t h) { return &h->noalloc_scratch; }

sa_status check_call(const char* fn, int B, int H, int L, int d, const float* lambda, sa_dtype dtype) {
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  return check_lambda(fn, lambda, H);
}

// The checks and the two launches of sa_rope_attn, with q', k' placed at caller-given
// device addresses instead of a workspace argument.
sa_status rope_attn_into(const char* fn, sa_attn_t h, const void* q, const void* k, const void* v,
                         const int32_t* positions, void* out, int B, int H, int L, int d,
                         int window, const float* lambda, sa_dtype dtype, void* q_rot, void* k_rot,
                         sa_stream_t stream) {
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q || !k || !v || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v and out must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v and out must be 16-byte aligned", fn);
  if (!aligned16(q_rot) || !aligned16(k_rot))
    return fail(SA_ERR_INVALID_ARG, "%s: the q' / k' scratch must be 16-byte aligned", fn);
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  if (dtype == SA_FP32) {
    // v^T follows k' (the caller's scratch holds all three)
    size_t n32 = 0;
    qk_elems(B, H, L, 2, &n32);
    void* v_t = static_cast<uint8_t*>(k_rot) + align256(n32 * 4);
    st = launch_rope_f32(h, q, k, positions, q_rot, k_rot, B, H, L, stream, v, v_t);
    if (st != SA_OK) return st;
    return launch_attn_f32(h, q_rot, k_rot, v_t, out, B, H, L, window, lambda, stream);
  }
  st = launch_rope(h, q, k, positions, q_rot, k_rot, B, H, L, diff ? 2 : 1, dtype, stream);
  if (st != SA_OK) return st;
  return launch_attn(h, q_rot, k_rot, v, out, B, H, L, window, lambda, dtype, nullptr, stream);
}

}  // namespace sa

extern "C" {

const char* sa_last_error(void) { return g_msg; }

const char* sa_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
    case SA_ERR_DEVICE_TIMEOUT: return "SA_ERR_DEVICE_TIMEOUT";
    case SA_ERR_NO_DEVICE: return "SA_ERR_NO_DEVICE";
    case SA_ERR_WORKSPACE: return "SA_ERR_WORKSPACE";
  }
  return "SA_ERR_UNKNOWN";
}

sa_status sa_attn_create(sa_attn_t* handle, int device, float rope_base) {
  if (!handle) return fail(SA_ERR_INVALID_ARG, "sa_attn_create: handle pointer is NULL");
  *handle = nullptr;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base))
    return fail(SA_ERR_INVALID_ARG, "sa_attn_create: rope_base must be finite and > 1 (got %g)",
                static_cast<double>(rope_base));
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || count == 0)
    return fail(SA_ERR_NO_DEVICE, "sa_attn_create: no CUDA device (%s)", cudaGetErrorString(e));
  if (device < 0 || device >= count)
    return fail(SA_ERR_NO_DEVICE, "sa_attn_create: device %d out of range [0, %d)", device, count);
  DeviceGuard guard(device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "sa_attn_create: cannot select device %d", device);
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, device)) != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_attn_create: %s", cudaGetErrorString(e));
  if (prop.major != 10 || prop.minor != 3)
    return fail(SA_ERR_UNSUPPORTED,
                "sa_attn_create: device %d is sm_%d%d; this library is built for sm_103a (GB300)",
                device, prop.major, prop.minor);

  sa_attn_s* h = new (std::nothrow) sa_attn_s();
  if (!h) return fail(SA_ERR_CUDA, "sa_attn_create: out of host memory");
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->rope_base = rope_base;
  h->timeout_ns = 1000000000ull;  // 1 s per pipeline wait
  for (int i = 0; i < sa::kHeadDim / 2; ++i)
    h->inv_freq[i] = static_cast<float>(
        std::pow(static_cast<double>(rope_base), -2.0 * i / static_cast<double>(sa::kHeadDim)));

  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    delete h;
    return fail(SA_ERR_CUDA, "sa_attn_create: cuTensorMapEncodeTiled unavailable (%s)",
                cudaGetErrorString(e));
  }
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  if ((e = cudaMalloc(&h->d_err, sizeof(int))) != cudaSuccess) {
    delete h;
    return fail(SA_ERR_CUDA, "sa_attn_create: cudaMalloc: %s", cudaGetErrorString(e));
  }
  for (int wq = 0; wq < 2; ++wq)
    for (int nm = 0; nm < 2; ++nm) h->rope_blocks_per_sm[wq][nm] = sa::rope_blocks_per_sm(wq != 0, nm != 0);
  h->host_ready = create_host_streams(h);
  create_table(h);
  if ((e = cudaMemset(h->d_err, 0, sizeof(int))) != cudaSuccess ||
      (e = sa::fmha_set_attributes()) != cudaSuccess || (e = sa::fmha_tf32_set_attributes()) != cudaSuccess ||
      (e = sa::fmha_swa_set_attributes()) != cudaSuccess) {
    cudaFree(h->d_err);
    destroy_host_streams(h);
    delete h;
    return fail(SA_ERR_CUDA, "sa_attn_create: %s", cudaGetErrorString(e));
  }
  int regs = -1, regs_tf32 = -1;
  if (!sa::fmha_check_registers(&regs) || !sa::fmha_tf32_check(&regs_tf32) || !sa::fmha_swa_check()) {
    // The warpgroup register split (setmaxnreg) is sized for this launch allocation; any
    // other value could make the register grow wait forever, so refuse to run.
    cudaFree(h->d_err);
    destroy_host_streams(h);
    delete h;
    return fail(SA_ERR_UNSUPPORTED, "sa_attn_create: attention kernel built with %d registers per "
                "thread (expected %d) or for an architecture other than sm_103a", regs, sa::kFmhaLaunchRegs);
  }
  *handle = h;
  return ok();
}

sa_status sa_attn_destroy(sa_attn_t h) {
  if (!h) return ok();
  {
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->d_err);
    destroy_host_streams(h);
  }
  delete h;
  return ok();
}

size_t sa_rope_table_bytes(int L) {
  if (L <= 0 || L >= sa::kMaxL) return 0;
  return static_cast<size_t>(L) * (sa::kHeadDim / 2) * 2 * sizeof(float);
}

size_t sa_rope_attn_workspace_size(int B, int H, int L, int d, int differential) {
  size_t n = 0;
  if (d != sa::kHeadDim || !qk_elems(B, H, L, differential ? 2 : 1, &n)) return 0;
  return align256(sa_rope_table_bytes(L)) + align256(n * 2) + split_bytes(B, H, L, differential != 0);
}

size_t sa_rope_attn_workspace_bytes(int B, int H, int L, int d, int differential, sa_dtype dtype) {
  if (dtype == SA_FP16 || dtype == SA_BF16) return sa_rope_attn_workspace_size(B, H, L, d, differential);
  if (dtype != SA_FP32 || !differential || d != sa::kHeadDim || L >= sa::kMaxL) return 0;
  return f32_ws_bytes(B, H, L);
}

size_t sa_attn_fwd_workspace_bytes(int B, int H, int L, int d, int differential, sa_dtype dtype) {
  if (dtype == SA_FP16 || dtype == SA_BF16) return sa_attn_fwd_workspace_size(B, H, L, d, differential);
  size_t n = 0;
  if (dtype != SA_FP32 || !differential || d != sa::kHeadDim || L >= sa::kMaxL || !qk_elems(B, H, L, 2, &n))
    return 0;
  return f32_vt_bytes(B, H, L);
}

size_t sa_attn_fwd_workspace_size(int B, int H, int L, int d, int differential) {
  size_t n = 0;
  if (d != sa::kHeadDim || !qk_elems(B, H, L, differential ? 2 : 1, &n)) return 0;
  return split_bytes(B, H, L, differential != 0);
}

sa_status sa_rope_qk(sa_attn_t h, const void* q, const void* k, const int32_t* positions,
                     void* q_rot, void* k_rot, int B, int H, int L, int d, int nmaps, sa_dtype dtype,
                     sa_stream_t stream) {
  const char* fn = "sa_rope_qk";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q || !k || !q_rot || !k_rot)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, q_rot and k_rot must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_rot) || !aligned16(k_rot))
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, q_rot and k_rot must be 16-byte aligned", fn);
  if (nmaps != 1 && nmaps != 2) return fail(SA_ERR_INVALID_ARG, "%s: nmaps must be 1 or 2", fn);
  sa_status st = check_shape(fn, B, H, L, d, dtype, nmaps == 2);
  if (st != SA_OK) return st;
  if (dtype == SA_FP32) return launch_rope_f32(h, q, k, positions, q_rot, k_rot, B, H, L, stream);
  return launch_rope(h, q, k, positions, q_rot, k_rot, B, H, L, nmaps, dtype, stream);
}

sa_status sa_attn_fwd(sa_attn_t h, const void* q_rot, const void* k_rot, const void* v, void* out,
                      int B, int H, int L, int d, int window, const float* lambda, sa_dtype dtype,
                      void* workspace, size_t workspace_bytes, sa_stream_t stream) {
  const char* fn = "sa_attn_fwd";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q_rot || !k_rot || !v || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q_rot, k_rot, v and out must be non-NULL", fn);
  if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return fail(SA_ERR_INVALID_ARG, "%s: q_rot, k_rot, v, out and workspace must be 16-byte aligned", fn);
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  if (dtype == SA_FP32) {
    // v^T (TF32) into the workspace, then attention on it
    if (!workspace || workspace_bytes < f32_vt_bytes(B, H, L))
      return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed for the FP32 form, %zu given%s", fn,
                  f32_vt_bytes(B, H, L), workspace_bytes, workspace ? "" : " (NULL)");
    st = launch_rope_f32(h, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, L, stream, v, workspace);
    if (st != SA_OK) return st;
    return launch_attn_f32(h, q_rot, k_rot, workspace, out, B, H, L, window, lambda, stream);
  }
  if (workspace && workspace_bytes < split_bytes(B, H, L, diff))
    return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn,
                split_bytes(B, H, L, diff), workspace_bytes);
  return launch_attn(h, q_rot, k_rot, v, out, B, H, L, window, lambda, dtype, workspace, stream);
}

sa_status sa_rope_k(sa_attn_t h, const void* k, const int32_t* positions, void* k_rot, void* cs_table,
                    int B, int H, int L, int d, int nmaps, sa_dtype dtype, sa_stream_t stream) {
  const char* fn = "sa_rope_k";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (reject_fp32(fn, dtype) != SA_OK) return SA_ERR_UNSUPPORTED;
  if (!k || !k_rot || !cs_table)
    return fail(SA_ERR_INVALID_ARG, "%s: k, k_rot and cs_table must be non-NULL", fn);
  if (!aligned16(k) || !aligned16(k_rot) || !aligned16(cs_table))
    return fail(SA_ERR_INVALID_ARG, "%s: k, k_rot and cs_table must be 16-byte aligned", fn);
  if (nmaps != 1 && nmaps != 2) return fail(SA_ERR_INVALID_ARG, "%s: nmaps must be 1 or 2", fn);
  sa_status st = check_shape(fn, B, H, L, d, dtype, nmaps == 2);
  if (st != SA_OK) return st;
  return launch_rope(h, nullptr, k, positions, nullptr, k_rot, B, H, L, nmaps, dtype, stream, cs_table);
}

sa_status sa_attn_fwd_rope_q(sa_attn_t h, const void* q, const void* k_rot, const void* cs_table,
                             const void* v, void* out, int B, int H, int L, int d, int window,
                             const float* lambda, sa_dtype dtype, void* workspace,
                             size_t workspace_bytes, sa_stream_t stream) {
  const char* fn = "sa_attn_fwd_rope_q";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (reject_fp32(fn, dtype) != SA_OK) return SA_ERR_UNSUPPORTED;
  if (!q || !k_rot || !cs_table || !v || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k_rot, cs_table, v and out must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k_rot) || !aligned16(cs_table) || !aligned16(v) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return fail(SA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  if (workspace && workspace_bytes < split_bytes(B, H, L, diff))
    return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn,
                split_bytes(B, H, L, diff), workspace_bytes);
  return launch_attn(h, q, k_rot, v, out, B, H, L, window, lambda, dtype, workspace, stream, cs_table);
}

}  // extern "C"

namespace {

// sa_rope_attn and sa_rope_attn_qknorm: checks, then the K pass (with the table) and the
// attention kernel (with the Q prologue), both on the caller's workspace.
// side_ok: the call may run its k pass on the SMs its attention grid leaves idle (false when
// other work of the same call runs beside it, as the chunks of the host-buffer call do).
sa_status rope_attn_ws(const char* fn, sa_attn_t h, const void* q, const void* k, const void* v,
                       const int32_t* positions, void* out, int B, int H, int L, int d, int window,
                       const float* lambda, sa_dtype dtype, void* workspace, size_t workspace_bytes,
                       sa_stream_t stream, const QkNorm* nrm, bool side_ok = true) {
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q || !k || !v || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v and out must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v, out and workspace must be 16-byte aligned", fn);
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  if (dtype == SA_FP32) {
    if (nrm) return fail(SA_ERR_UNSUPPORTED, "%s: the QK-RMSNorm form takes SA_FP16 or SA_BF16", fn);
    const size_t need32 = f32_ws_bytes(B, H, L);
    if (!workspace || workspace_bytes < need32)
      return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given%s", fn, need32,
                  workspace_bytes, workspace ? "" : " (NULL)");
    size_t n32 = 0;
    qk_elems(B, H, L, 2, &n32);
    uint8_t* ws32 = static_cast<uint8_t*>(workspace);
    uint8_t* k32 = ws32 + align256(n32 * 4);
    uint8_t* vt32 = k32 + align256(n32 * 4);
    st = launch_rope_f32(h, q, k, positions, ws32, k32, B, H, L, stream, v, vt32);
    if (st != SA_OK) return st;
    return launch_attn_f32(h, ws32, k32, vt32, out, B, H, L, window, lambda, stream);
  }
  const size_t need = sa_rope_attn_workspace_size(B, H, L, d, diff);
  if (!workspace || workspace_bytes < need)
    return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given%s", fn, need,
                workspace_bytes, workspace ? "" : " (NULL)");
  // workspace: the (cos, sin) table, k', the split region.  The RoPE pass rotates k and writes
  // the table; the attention kernel rotates q in its prologue.
  const size_t nqk = static_cast<size_t>(B) * H * (diff ? 2 : 1) * L * sa::kHeadDim;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* cs = ws;
  void* k_rot = ws + align256(sa_rope_table_bytes(L));
  void* split_ws = static_cast<uint8_t*>(k_rot) + align256(nqk * 2);
  const int side = side_ok && positions == nullptr && h->d_cs != nullptr && L <= h->cs_cap
                       ? side_sms(h, attn_grid(h, B, H, L, window, diff, true).ctas, static_cast<long long>(nqk) * 2)
                       : 0;
  if (side > 0) {
    // A grid that leaves SMs idle, default positions: the pass runs on the idle SMs and writes
    // no table, the prologue reads the handle's, and the attention CTAs start at once on the
    // other SMs (only their K loads wait for the pass).  Larger grids keep the per-call table,
    // which the pass leaves in L2 right before the prologue reads it.
    st = launch_rope(h, nullptr, k, nullptr, nullptr, k_rot, B, H, L, diff ? 2 : 1, dtype, stream, nullptr, nrm,
                     side);
    if (st != SA_OK) return st;
    return launch_attn(h, q, k_rot, v, out, B, H, L, window, lambda, dtype, split_ws, stream, h->d_cs, nrm,
                       h->cs_cap, true);
  }
  st = launch_rope(h, nullptr, k, positions, nullptr, k_rot, B, H, L, diff ? 2 : 1, dtype, stream, cs, nrm);
  if (st != SA_OK) return st;
  return launch_attn(h, q, k_rot, v, out, B, H, L, window, lambda, dtype, split_ws, stream, cs, nrm);
}

}  // namespace

extern "C" {

sa_status sa_rope_attn(sa_attn_t h, const void* q, const void* k, const void* v,
                       const int32_t* positions, void* out, int B, int H, int L, int d, int window,
                       const float* lambda, sa_dtype dtype, void* workspace,
                       size_t workspace_bytes, sa_stream_t stream) {
  return rope_attn_ws("sa_rope_attn", h, q, k, v, positions, out, B, H, L, d, window, lambda, dtype,
                      workspace, workspace_bytes, stream, nullptr);
}

sa_status sa_rope_attn_qknorm(sa_attn_t h, const void* q, const void* k, const void* v,
                              const int32_t* positions, const float* gamma_q, const float* gamma_k,
                              float eps, void* out, int B, int H, int L, int d, int window,
                              const float* lambda, sa_dtype dtype, void* workspace,
                              size_t workspace_bytes, sa_stream_t stream) {
  const char* fn = "sa_rope_attn_qknorm";
  QkNorm nrm;
  sa_status st = make_qknorm(fn, gamma_q, gamma_k, eps, &nrm);
  if (st != SA_OK) return st;
  return rope_attn_ws(fn, h, q, k, v, positions, out, B, H, L, d, window, lambda, dtype, workspace,
                      workspace_bytes, stream, &nrm);
}

}  // extern "C"

// ---------------------------------------------------------------- host buffers

namespace {

// Chunks of sa_rope_attn_host: contiguous ranges of the B*H (batch, head) planes, at most
// kHostChunks at a time in flight and at most kMaxDiffHeads planes each.  Every copy has a
// fixed cost, so a chunk carries at least kHostChunkBytes of copies where the sizes allow;
// copies of at least half that are still cut in two, so that one half's copies overlap the
// other half's computation (measured: 94 -> 91 us per call at 10.6 MB of copies, while
// 4 MiB chunks everywhere were slower at 50 MB).
constexpr double kHostChunkBytes = 16.0 * 1024 * 1024;

struct HostChunks {
  long long planes;
  int n;          // chunks
  int max_len;    // planes in the largest chunk
  long long first(int c) const { return c * planes / n; }
  int len(int c) const { return static_cast<int>(first(c + 1) - first(c)); }
};

HostChunks host_chunks(int B, int H, int L, bool diff) {
  HostChunks hc;
  hc.planes = static_cast<long long>(B) * H;
  // bytes copied per plane: q, k (both maps), v in and out out
  const double plane_bytes = 2.0 * L * sa::kHeadDim * (diff ? 2 : 1) * 4;
  const double total = hc.planes * plane_bytes;
  const long long by_size = total >= kHostChunkBytes ? static_cast<long long>(total / kHostChunkBytes)
                            : (total >= kHostChunkBytes / 2 ? 2 : 1);
  long long n = std::min<long long>(std::min<long long>(sa::kHostChunks, by_size), hc.planes);
  n = std::max<long long>(n, (hc.planes + sa::kMaxDiffHeads - 1) / sa::kMaxDiffHeads);
  hc.n = static_cast<int>(n);
  hc.max_len = static_cast<int>((hc.planes + n - 1) / n);
  return hc;
}

// Device bytes of sa_rope_attn_host: q, k, v, out, then one sa_rope_attn workspace per compute
// stream (for its largest chunk).
size_t host_ws_bytes(int B, int H, int L, int d, bool diff, size_t* per_chunk) {
  size_t nqk = 0;
  if (d != sa::kHeadDim || !qk_elems(B, H, L, diff ? 2 : 1, &nqk)) return 0;
  const HostChunks hc = host_chunks(B, H, L, diff);
  const size_t nv = static_cast<size_t>(B) * H * L * (diff ? 2 : 1) * sa::kHeadDim;
  const size_t chunk = sa_rope_attn_workspace_size(1, hc.max_len, L, d, diff);
  if (chunk == 0) return 0;
  if (per_chunk) *per_chunk = chunk;
  return 2 * align256(nqk * 2) + 2 * align256(nv * 2) +
         static_cast<size_t>(std::min(hc.n, sa::kHostChunks)) * chunk;
}

}  // namespace

extern "C" {

size_t sa_rope_attn_host_workspace_size(int B, int H, int L, int d, int differential) {
  if (B <= 0 || H <= 0 || L <= 0 || L >= sa::kMaxL) return 0;
  return host_ws_bytes(B, H, L, d, differential != 0, nullptr);
}

sa_status sa_rope_attn_host(sa_attn_t h, const void* q, const void* k, const void* v,
                            const int32_t* positions, void* out, int B, int H, int L, int d,
                            int window, const float* lambda, sa_dtype dtype, void* workspace,
                            size_t workspace_bytes, sa_stream_t stream) {
  const char* fn = "sa_rope_attn_host";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (reject_fp32(fn, dtype) != SA_OK) return SA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v and out must be non-NULL", fn);
  if (!workspace || !aligned16(workspace))
    return fail(SA_ERR_INVALID_ARG, "%s: workspace must be a 16-byte aligned device pointer", fn);
  const bool diff = lambda != nullptr;
  sa_status st = check_shape(fn, B, H, L, d, dtype, diff);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  size_t per_chunk = 0;
  const size_t need = host_ws_bytes(B, H, L, d, diff, &per_chunk);
  if (workspace_bytes < need)
    return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need, workspace_bytes);
  if (!h->host_ready) return fail(SA_ERR_CUDA, "%s: the handle's copy streams could not be created", fn);
  DeviceGuard guard(h->device);
  if (!guard.ok) return fail(SA_ERR_CUDA, "cannot select device %d", h->device);

  // per plane: q/k elements (both maps for the differential form) and v/out elements
  const size_t pqk = static_cast<size_t>(diff ? 2 : 1) * L * sa::kHeadDim;
  const size_t pv = static_cast<size_t>(L) * (diff ? 2 : 1) * sa::kHeadDim;
  const size_t nqk = static_cast<size_t>(B) * H * pqk, nv = static_cast<size_t>(B) * H * pv;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dq = ws;
  uint8_t* dk = dq + align256(nqk * 2);
  uint8_t* dv = dk + align256(nqk * 2);
  uint8_t* dout = dv + align256(nv * 2);
  uint8_t* regions = dout + align256(nv * 2);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  const HostChunks hc = host_chunks(B, H, L, diff);
  if (hc.n == 1) {
    // one chunk: nothing to overlap, so everything goes on `stream` in order
    cudaError_t e = cudaMemcpyAsync(dq, q, nqk * 2, cudaMemcpyHostToDevice, cs);
    e = e != cudaSuccess ? e : cudaMemcpyAsync(dk, k, nqk * 2, cudaMemcpyHostToDevice, cs);
    e = e != cudaSuccess ? e : cudaMemcpyAsync(dv, v, nv * 2, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: copy in: %s", fn, cudaGetErrorString(e));
    st = rope_attn_ws(fn, h, dq, dk, dv, positions, dout, B, H, L, d, window, lambda, dtype, regions,
                      per_chunk, stream, nullptr);
    if (st != SA_OK) return st;
    e = cudaMemcpyAsync(out, dout, nv * 2, cudaMemcpyDeviceToHost, cs);
    if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: copy out: %s", fn, cudaGetErrorString(e));
    return ok();
  }
  // The caller's earlier work on `stream` comes first; every internal stream starts after it.
  cudaError_t e = cudaEventRecord(h->he_entry, cs);
  e = e != cudaSuccess ? e : cudaStreamWaitEvent(h->hs_in, h->he_entry, 0);
  e = e != cudaSuccess ? e : cudaStreamWaitEvent(h->hs_out, h->he_entry, 0);
  for (int c = 0; c < sa::kHostChunks && e == cudaSuccess; ++c) e = cudaStreamWaitEvent(h->hs_comp[c], h->he_entry, 0);
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));

  // Chunk c: copy its planes in (copy stream), RoPE + attention on compute stream c % kHostChunks
  // (chunks on different streams run side by side), copy its output back (output stream).
  for (int c = 0; c < hc.n; ++c) {
    const long long p0 = hc.first(c);
    const int len = hc.len(c);
    const int slot = c % sa::kHostChunks;
    const size_t oqk = static_cast<size_t>(p0) * pqk * 2, ov = static_cast<size_t>(p0) * pv * 2;
    const size_t bqk = static_cast<size_t>(len) * pqk * 2, bv = static_cast<size_t>(len) * pv * 2;
    e = cudaMemcpyAsync(dq + oqk, static_cast<const uint8_t*>(q) + oqk, bqk, cudaMemcpyHostToDevice, h->hs_in);
    e = e != cudaSuccess ? e : cudaMemcpyAsync(dk + oqk, static_cast<const uint8_t*>(k) + oqk, bqk, cudaMemcpyHostToDevice, h->hs_in);
    e = e != cudaSuccess ? e : cudaMemcpyAsync(dv + ov, static_cast<const uint8_t*>(v) + ov, bv, cudaMemcpyHostToDevice, h->hs_in);
    e = e != cudaSuccess ? e : cudaEventRecord(h->he_in[slot], h->hs_in);
    e = e != cudaSuccess ? e : cudaStreamWaitEvent(h->hs_comp[slot], h->he_in[slot], 0);
    if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: copy in: %s", fn, cudaGetErrorString(e));
    float lam[sa::kMaxDiffHeads];
    if (diff)
      for (int i = 0; i < len; ++i) lam[i] = lambda[(p0 + i) % H];
    st = rope_attn_ws(fn, h, dq + oqk, dk + oqk, dv + ov, positions, dout + ov, 1, len, L, d, window,
                      diff ? lam : nullptr, dtype, regions + slot * per_chunk, per_chunk, h->hs_comp[slot], nullptr,
                      false);
    if (st != SA_OK) return st;
    e = cudaEventRecord(h->he_done[slot], h->hs_comp[slot]);
    e = e != cudaSuccess ? e : cudaStreamWaitEvent(h->hs_out, h->he_done[slot], 0);
    e = e != cudaSuccess ? e : cudaMemcpyAsync(static_cast<uint8_t*>(out) + ov, dout + ov, bv, cudaMemcpyDeviceToHost, h->hs_out);
    if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: copy out: %s", fn, cudaGetErrorString(e));
  }
  // `stream` continues once the last output copy is done.
  e = cudaEventRecord(h->he_exit, h->hs_out);
  e = e != cudaSuccess ? e : cudaStreamWaitEvent(cs, h->he_exit, 0);
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return ok();
}

}  // extern "C"

extern "C" {

sa_status sa_qknorm_rope_qk(sa_attn_t h, const void* q, const void* k, const int32_t* positions,
                            const float* gamma_q, const float* gamma_k, float eps, void* q_rot,
                            void* k_rot, int B, int H, int L, int d, int nmaps, sa_dtype dtype,
                            sa_stream_t stream) {
  const char* fn = "sa_qknorm_rope_qk";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (reject_fp32(fn, dtype) != SA_OK) return SA_ERR_UNSUPPORTED;
  if (!q || !k || !q_rot || !k_rot)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, q_rot and k_rot must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_rot) || !aligned16(k_rot))
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, q_rot and k_rot must be 16-byte aligned", fn);
  if (nmaps != 1 && nmaps != 2) return fail(SA_ERR_INVALID_ARG, "%s: nmaps must be 1 or 2", fn);
  sa_status st = check_shape(fn, B, H, L, d, dtype, nmaps == 2);
  if (st != SA_OK) return st;
  QkNorm nrm;
  if ((st = make_qknorm(fn, gamma_q, gamma_k, eps, &nrm)) != SA_OK) return st;
  return launch_rope(h, q, k, positions, q_rot, k_rot, B, H, L, nmaps, dtype, stream, nullptr, &nrm);
}

sa_status sa_rope_qkv_f32(sa_attn_t h, const void* q, const void* k, const void* v, const int32_t* positions,
                         void* q_rot, void* k_rot, void* v_t, int B, int H, int L, int d, sa_stream_t stream) {
  const char* fn = "sa_rope_qkv_f32";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q || !k || !v || !q_rot || !k_rot || !v_t)
    return fail(SA_ERR_INVALID_ARG, "%s: q, k, v, q_rot, k_rot and v_t must be non-NULL", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v_t))
    return fail(SA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  sa_status st = check_shape(fn, B, H, L, d, SA_FP32, true);
  if (st != SA_OK) return st;
  return launch_rope_f32(h, q, k, positions, q_rot, k_rot, B, H, L, stream, v, v_t);
}

sa_status sa_attn_fwd_f32(sa_attn_t h, const void* q_rot, const void* k_rot, const void* v_t, void* out, int B,
                          int H, int L, int d, int window, const float* lambda, sa_stream_t stream) {
  const char* fn = "sa_attn_fwd_f32";
  if (!h) return fail(SA_ERR_INVALID_ARG, "%s: handle is NULL", fn);
  if (!q_rot || !k_rot || !v_t || !out)
    return fail(SA_ERR_INVALID_ARG, "%s: q_rot, k_rot, v_t and out must be non-NULL", fn);
  if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v_t) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  if (!lambda) return fail(SA_ERR_UNSUPPORTED, "%s: the FP32 form is differential attention (lambda != NULL)", fn);
  sa_status st = check_shape(fn, B, H, L, d, SA_FP32, true);
  if (st != SA_OK) return st;
  if ((st = check_lambda(fn, lambda, H)) != SA_OK) return st;
  return launch_attn_f32(h, q_rot, k_rot, v_t, out, B, H, L, window, lambda, stream);
}

sa_status sa_attn_set_timeout(sa_attn_t h, unsigned long long timeout_ns) {
  if (!h) return fail(SA_ERR_INVALID_ARG, "sa_attn_set_timeout: handle is NULL");
  if (timeout_ns < 100)
    return fail(SA_ERR_INVALID_ARG, "sa_attn_set_timeout: limit must be at least 100 ns");
  h->timeout_ns = timeout_ns;
  return ok();
}

sa_status sa_attn_check(sa_attn_t h) {
  if (!h) return fail(SA_ERR_INVALID_ARG, "sa_attn_check: handle is NULL");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "sa_attn_check: %s", cudaGetErrorString(e));
  int word = 0;
  if ((e = cudaMemcpy(&word, h->d_err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemset(h->d_err, 0, sizeof(int))) != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_attn_check: %s", cudaGetErrorString(e));
  if (word != 0)
    return fail(SA_ERR_DEVICE_TIMEOUT,
                "sa_attn_check: a kernel gave up on a pipeline wait (error bits 0x%x: 1 = TMA, "
                "2 = MMA, 4 = softmax)",
                word);
  return ok();
}

}  // extern "C"
