// ssd_noalloc.cu -- ssd_chunk_scan_fwd_noalloc: the CUDA-core chunked
// forward with its scratch memory in a fixed array compiled into the
// library, for callers that cannot allocate device memory (contract in
// include/ssd.h).
#include <cuda_runtime.h>

#include <mutex>

#include "ssd.h"
#include "ssd_internal.h"

namespace {

// Upper bound on the scratch one call may use.  The array lives in every
// device's global memory from the moment the library is loaded on that
// device until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device.  In host code the
// name g_scratch is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
ssd_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" ssd_status_t ssd_chunk_scan_fwd_noalloc(
    const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
    int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups, int chunk_size,
    ssd_dtype_t in_dtype, const float* init_states, const int32_t* cu_seqlens, int nseq,
    float* y, float* final_states, int32_t* dev_status, void* stream) {
  ssd::FwdArgs a{};
  a.x = x;
  a.dt = dt;
  a.A = A;
  a.B = B;
  a.C = C;
  a.D = D;
  a.batch = batch;
  a.seqlen = seqlen;
  a.H = nheads;
  a.P = headdim;
  a.N = dstate;
  a.G = ngroups;
  a.Q = chunk_size;
  a.dtype = in_dtype;
  a.init = init_states;
  a.cu = cu_seqlens;
  a.nseq = cu_seqlens ? nseq : batch;
  a.y = y;
  a.final_states = final_states;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  ssd_status_t st = ssd::check_fwd_args(a, true);
  if (st != SSD_OK) return st;
  if (ssd::simt_workspace_bytes(a) > kScratchBytes) return SSD_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != SSD_OK) return st;
  a.ws = scratch;
  a.ws_bytes = kScratchBytes;
  if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), a.stream) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (a.nseq == 0) return SSD_OK;
  return ssd::simt_forward(a);
}
