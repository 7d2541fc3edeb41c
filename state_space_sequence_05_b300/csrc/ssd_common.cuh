// ssd_common.cuh -- helpers shared by the library's CUDA sources.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// Input element loads (x, dt, B, C arrive as float32 or bfloat16).
__device__ __forceinline__ float ld_in(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p)));
}

// Device-side error report: the first error wins.
__device__ __forceinline__ void report(int32_t* dev_status, int code) {
  if (dev_status) atomicCAS(reinterpret_cast<int*>(dev_status), 0, code);
}

// Sequence bookkeeping shared by the forward kernels.  A "sequence" is a
// batch row (rows of `seqlen` tokens) or a packed cu_seqlens range; tokens
// are indexed in the flattened [batch*seqlen] token space.
struct SeqInfo {
  const int32_t* cu;  // device cu_seqlens or nullptr (batch mode)
  int seqlen;         // tokens per row (batch mode)
  int nseq;           // sequences
  __device__ __forceinline__ long long begin(int s) const {
    return cu ? (long long)cu[s] : (long long)s * seqlen;
  }
  __device__ __forceinline__ long long end(int s) const {
    return cu ? (long long)cu[s + 1] : (long long)(s + 1) * seqlen;
  }
};

// Largest s with offs[s] <= g, over offs[0..n] (non-decreasing, offs[0]=0).
__device__ __forceinline__ int upper_index(const int32_t* offs, int n, int g) {
  int lo = 0, hi = n;  // invariant: offs[lo] <= g < offs[hi] (when g < offs[n])
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (offs[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

constexpr int kMaxSeqChunksBlock = 1024;

}  // namespace ssd
