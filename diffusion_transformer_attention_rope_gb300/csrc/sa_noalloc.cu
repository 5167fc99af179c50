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
// with cudaGetSymbolAddress, with the device current, once per device, on the first call made on
// that device (that first call should therefore come before any stream capture).  All calls share
// the one array: calls that can overlap on the GPU (different streams, no ordering) race on it.
// Nothing in it has to start at zero: the RoPE stage overwrites every byte a call then reads.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sa_attn.h"
#include "sa_kernels.h"

namespace {

constexpr size_t kScratchBytes = SA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of g_scratch on `device`, looked up once with that device current.
sa_status scratch_address(int device, void** addr) {
  if (device < 0 || device >= kMaxDevices)
    return sa::set_error(SA_ERR_UNSUPPORTED, "sa_rope_attn_noalloc: device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[device]) {
    *addr = g_scratch_addr[device];
    return SA_OK;
  }
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
  g_scratch_addr[device] = p;
  *addr = p;
  return SA_OK;
}

}  // namespace

extern "C" sa_status sa_rope_attn_noalloc(sa_attn_t h, const void* q, const void* k, const void* v,
                                          const int32_t* positions, void* out, int B, int H, int L,
                                          int d, int window, const float* lambda, sa_dtype dtype,
                                          sa_stream_t stream) {
  if (!h) return sa::set_error(SA_ERR_INVALID_ARG, "sa_rope_attn_noalloc: handle is NULL");
  const bool diff = lambda != nullptr;
  if (sa_rope_attn_workspace_size(B, H, L, d, diff ? 1 : 0) == 0)
    return sa::set_error(SA_ERR_INVALID_ARG, "sa_rope_attn_noalloc: invalid sizes (B, H, L >= 1, d = 64)");
  // The scratch holds q' and k' only: this entry point runs the attention stage without the
  // split region (one CTA per query block).
  const size_t nqk = static_cast<size_t>(B) * H * (diff ? 2 : 1) * L * d;
  const size_t need = 2 * round256(nqk * 2);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "sa_rope_attn_noalloc: this shape needs %zu bytes of scratch but the built-in scratch "
             "holds %zu (SA_NOALLOC_SCRATCH_BYTES); use sa_rope_attn with a workspace",
             need, kScratchBytes);
    return sa::set_error(SA_ERR_WORKSPACE, msg);
  }
  void* base = nullptr;
  const sa_status st = scratch_address(sa::handle_device(h), &base);
  if (st != SA_OK) return st;
  unsigned char* ws = static_cast<unsigned char*>(base);
  return sa::rope_attn_into("sa_rope_attn_noalloc", h, q, k, v, positions, out, B, H, L, d, window,
                            lambda, dtype, ws, ws + round256(nqk * 2), stream);
}
