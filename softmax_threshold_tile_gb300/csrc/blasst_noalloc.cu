// The host-buffer call without any allocation (blasst_attn_fwd_host_noalloc in blasst.h): its
// device workspace is a fixed-size array of this library instead of a caller's buffer. This
// file holds the array, looks up its device address once per device, and hands that address to
// the head-group pipeline of blasst_attn_fwd_host as the workspace.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "blasst.h"
#include "blasst_internal.h"

namespace blasst {
namespace {

constexpr size_t kScratchBytes = BLASST_NOALLOC_SCRATCH_BYTES;

// The workspace of every blasst_attn_fwd_host_noalloc call on a device. In host code this name
// only stands for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];  // the array's device address on each device, once looked up

// The array's device address on the current device, looked up on the first call there.
blasst_status scratch_address(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BLASST_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return BLASST_ERR_LAUNCH;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return BLASST_OK;
}

}  // namespace
}  // namespace blasst

extern "C" blasst_status blasst_attn_fwd_host_noalloc(const blasst_host_args* args) {
  // ---- argument checks: no CUDA call happens before all of them pass
  if (!args || args->struct_size != sizeof(blasst_host_args)) return BLASST_ERR_INVALID_ARG;
  blasst_host_args a = *args;
  if (a.workspace || a.workspace_bytes) return BLASST_ERR_INVALID_ARG;  // the library's buffer is used
  if (!a.q || !a.k || !a.v || !a.o || a.d != 128) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(a.scale) || !(a.scale > 0.f) || !std::isfinite(a.factor) || !(a.factor >= 0.f))
    return BLASST_ERR_INVALID_ARG;
  if (a.heads_per_group < 1 || a.heads_per_group > a.H) return BLASST_ERR_INVALID_ARG;
  const size_t one_head = blasst_host_workspace_bytes(a.B, a.H, a.Sq, a.Sk, 1);
  if (one_head == 0) return BLASST_ERR_INVALID_ARG;
  if (one_head > blasst::kScratchBytes) return BLASST_ERR_TOO_LARGE;
  // The largest head group, up to the one asked for, whose two slots fit the array.
  int hg = a.heads_per_group;
  while (hg > 1 && blasst_host_workspace_bytes(a.B, a.H, a.Sq, a.Sk, hg) > blasst::kScratchBytes) --hg;

  const blasst_status ds = blasst::check_device();
  if (ds != BLASST_OK) return ds;
  void* ws = nullptr;
  const blasst_status ss = blasst::scratch_address(&ws);
  if (ss != BLASST_OK) return ss;
  a.workspace = ws;
  a.workspace_bytes = blasst::kScratchBytes;
  a.heads_per_group = hg;
  return blasst::run_host_pipeline(a);
}
