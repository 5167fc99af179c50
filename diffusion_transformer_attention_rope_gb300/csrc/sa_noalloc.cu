// sa_noalloc.cu -- sa_rope_attn_noalloc: the full RoPE + attention call for callers that
// cannot allocate device memory.
//
// Some callers have inputs and outputs but no way to get scratch: a plugin whose enqueue hook
// receives only tensor pointers and a stream, a real-time audio thread that must never block in
// the allocator, or a process whose device memory is owned by another allocator.  For them the
// scratch that sa_rope_attn takes as `workspace` (the rotated q', k') lives here instead, in one
// file-scope device array of SA_NOALLOC_SCRATCH_BYTES.  Every GPU that loads this library keeps
// that array until the process exits.
//
// The array's name is only a host-side stand-in in host code, so its device address is looked up
// with cudaGetSymbolAddress, with the handle's device current, on the handle's first call of this
// entry point, and kept in the handle (that first call should therefore come before any stream
// capture).  A handle created after the context was torn down and made again looks the address up
// afresh.  All calls share the one array: calls that can overlap on the GPU (different streams, no
// ordering) race on it.  Nothing in it has to start at zero: the RoPE stage overwrites every byte
// a call then reads.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sa_attn.h"
#include "sa_kernels.h"

namespace {

constexpr size_t kScratchBytes = SA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of g_scratch in the context of the handle's device, looked up on the handle's
// first call (with that device current) and kept in the handle.
sa_status scratch_address(sa_attn_t h, void** addr) {
  std::lock_guard<std::mutex> lock(g_mu);
  void** slot = sa::handle_noalloc_slot(h);
  if (*slot) {
    *addr = *slot;
    return SA_OK;
  }
  const int device = sa::handle_device(h);
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess)
    return sa::set_error(SA_ERR_CUDA, "sa_rope_attn_noalloc: cudaGetDevice failed");
  if (prev != device && cudaSetDevice(device) != cudaSuccess)
    return sa::set_error(SA_ERR_CUDA, "sa_rope_attn_noalloc: cannot select the handle's device");
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess || !p) {
    char msg[256];
    snprintf(msg, sizeof(msg), "sa_rope_attn_noalloc: cudaGetSymbolAddress of the scratch array: %s",
             cudaGetErrorString(e));
    return sa::set_error(SA_ERR_CUDA, msg);
  }
  *slot = p;
  *addr = p;
  return SA_OK;
}

}  // namespace

extern "C" sa_status sa_rope_attn_noalloc(sa_attn_t h, const void* q, const void* k, const void* v,
                                          const int32_t* positions, void* out, int B, int H, int L,
                                          int d, int window, const float* lambda, sa_dtype dtype,
                                          sa_stream_t stream) {
  const char* fn = "sa_rope_attn_noalloc";
  if (!h) return sa::set_error(SA_ERR_INVALID_ARG, "sa_rope_attn_noalloc: handle is NULL");
  // sa_rope_attn's checks in its order (pointers, alignment, shape and dtype, lambda), then the
  // scratch size
  if (!q || !k || !v || !out)
    return sa::set_error(SA_ERR_INVALID_ARG, "sa_rope_attn_noalloc: q, k, v and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return sa::set_error(SA_ERR_INVALID_ARG, "sa_rope_attn_noalloc: q, k, v and out must be 16-byte aligned");
  sa_status st = sa::check_call(fn, B, H, L, d, lambda, dtype);
  if (st != SA_OK) return st;
  // The scratch holds q' and k' only: this entry point runs the attention stage without the
  // split region (one CTA per query block).
  const bool diff = lambda != nullptr;
  const size_t nqk = static_cast<size_t>(B) * H * (diff ? 2 : 1) * L * d;
  const size_t elem = dtype == SA_FP32 ? 4 : 2;
  // the FP32 form also keeps a transposed copy of v (128 rows of L rounded up to 4 keys)
  const size_t vt = dtype == SA_FP32 ? round256(static_cast<size_t>(B) * H * 2 * d * ((L + 3) & ~3) * 4) : 0;
  const size_t need = 2 * round256(nqk * elem) + vt;
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "sa_rope_attn_noalloc: this shape needs %zu bytes of scratch but the built-in scratch "
             "holds %zu (SA_NOALLOC_SCRATCH_BYTES); use sa_rope_attn with a workspace",
             need, kScratchBytes);
    return sa::set_error(SA_ERR_WORKSPACE, msg);
  }
  void* base = nullptr;
  st = scratch_address(h, &base);
  if (st != SA_OK) return st;
  unsigned char* ws = static_cast<unsigned char*>(base);
  return sa::rope_attn_into(fn, h, q, k, v, positions, out, B, H, L, d, window, lambda, dtype, ws,
                            ws + round256(nqk * elem), stream);
}
