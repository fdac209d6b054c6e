// fd_decode_attn_noalloc: the whole decode-attention hot path without any
// device allocation.
//
// Who needs it: a caller that must not allocate device memory while it runs.
// Typical cases are a plugin or custom op inside a serving framework whose own
// memory pool owns the device and forbids (or cannot account for) cudaMalloc
// from extensions, and latency-critical decode loops, where cudaMalloc may
// synchronise the whole device or fail under memory pressure in the middle of
// a step. fd_decode_attn allocates its workspace on first use and
// fd_decode_attn_ex needs the caller to provide one; this entry point needs
// neither: the split partials live in a fixed array compiled into the library.
//
// The array, g_noalloc_scratch, is a file-scope __device__ variable of
// FD_NOALLOC_SCRATCH_BYTES (32 MiB). Every device on which this library's code
// is loaded holds those 32 MiB until the process exits. In host code the
// array's name is only a host-side stand-in, not a device address, so it is
// never handed to a kernel: the device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
//
// The scratch starts with a fixed 64 KB region that holds only the counters
// a plan keeps at the head of its workspace (one split counter per (sequence,
// KV head), plus a work counter for a persistent grid), then the partials.
// Each call hands fd_decode_attn_ex a workspace that begins inside that region
// so that its counters end exactly where the region ends: partials of one
// shape can then never land on another shape's counters. The set-up of a
// device clears the whole array once, on the caller's stream, and waits for
// that stream, so the clear has finished before any later call on any stream
// runs; every completed call leaves its counters at zero again, and every
// partial a call reads was written earlier in the same call, so nothing is
// cleared between calls although each call finds the previous call's contents
// there. A call that fails part-way (a launch error, or a device wait that
// gave up) may leave a counter non-zero: fd_release makes the next call on
// each device run the set-up, and so the clear, again. All calls on a device
// share the one array, so calls that overlap on the GPU (on different streams,
// or from different threads) race on it and must be serialised by the caller.

#include <map>
#include <mutex>

#include <cuda_runtime.h>

#include "fd_decode_attn.h"
#include "fd_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[FD_NOALLOC_SCRATCH_BYTES];

constexpr size_t kCounterRegion = 64u << 10;  // split counters of up to 16384 groups

std::mutex g_scratch_mu;
std::map<int, void*> g_scratch_addr;  // device -> device address of the array

// Device address of the scratch array on `device`, which must be the current
// device. The first call for a device performs the lookup (and, with lazy
// module loading, loads this module on that device), clears the array on
// `stream` and waits for that stream; later calls return the cached address.
int scratch_address(int device, cudaStream_t stream, void** ptr) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  auto it = g_scratch_addr.find(device);
  if (it != g_scratch_addr.end()) {
    *ptr = it->second;
    return FD_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FD_ERR_CUDA;
  // The counters at the head of the scratch must start at zero (every
  // completed call leaves them zero again). The clear goes on the caller's
  // stream, ahead of this call's kernels, and the wait makes it finished for
  // calls on every other stream too.
  if (cudaMemsetAsync(p, 0, FD_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess) return FD_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FD_ERR_CUDA;
  g_scratch_addr[device] = p;
  *ptr = p;
  return FD_OK;
}

}  // namespace

namespace fd {

// Forget every device's set-up, so the next call on each device looks the
// address up and clears the array again (called by fd_release).
void noalloc_forget() {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  g_scratch_addr.clear();
}

}  // namespace fd

extern "C" int fd_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, void* out,
                                      const int* lens, int B, int NH, int NKV, int HS, int capacity,
                                      int window, float scale, fd_stream_t stream) {
  fd_plan_t plan;
  // Shape errors first, before any CUDA call (the SM count here is a dummy).
  int rc = fd_plan_sms(B, NH, NKV, HS, capacity, window, 0, 1, 1, 1, &plan);
  if (rc != FD_OK) return rc;
  if (B == 0) return FD_OK;
  if (!q || !k_cache || !v_cache || !out || !lens) return FD_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FD_ERR_CUDA;
  rc = fd_plan(B, NH, NKV, HS, capacity, window, 0, device, &plan);
  if (rc != FD_OK) return rc;
  const size_t counters = plan.workspace_zero_bytes;
  if (counters > kCounterRegion ||
      plan.workspace_bytes - counters > FD_NOALLOC_SCRATCH_BYTES - kCounterRegion)
    return FD_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  if (plan.workspace_bytes > 0) {
    void* base = nullptr;
    rc = scratch_address(device, reinterpret_cast<cudaStream_t>(stream), &base);
    if (rc != FD_OK) return rc;
    ws = static_cast<unsigned char*>(base) + (kCounterRegion - counters);
  }
  return fd_decode_attn_ex(&plan, ws, plan.workspace_bytes, nullptr, q, k_cache, v_cache, out, lens, B, NH, NKV,
                           HS, capacity, window, scale, stream);
}
