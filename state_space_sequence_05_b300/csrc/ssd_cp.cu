// ssd_cp.cu -- the two device steps of context (sequence) parallelism: a
// sequence cut into R consecutive slices, one per device, each slice run from
// a zero state; the state entering slice r is then the composition of the
// earlier slices' affine maps h -> exp(a_k) h + S_k (the composition rule
// (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2) of the Mamba paper review,
// feghi.github.io, sec. 4, applied to whole slices; the SSD review,
// dimensionstp.github.io, sec. 3-2 (4), passes states between chunks the
// same way).
//
//  * segment_decay_kernel: a[b, h] = sum_t dt[b, t, h] * A[h] over a slice
//    (the log of the slice's total decay), one block per (b, h).
//  * segment_combine_kernel: h_in[0] = init, h_in[r + 1] = exp(a[r]) h_in[r] +
//    S[r] for every (b, h, p, n), one thread per element, r walked in order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) segment_decay_kernel(const void* dt, const float* A,
                                                            int T, int H, float* a) {
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  float acc = 0.f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const long long i = ((long long)b * T + t) * H + h;
    acc += BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(dt)[i])
                : reinterpret_cast<const float*>(dt)[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
    a[bh] = s * A[h];
  }
}

__global__ void __launch_bounds__(256) segment_combine_kernel(const float* a, const float* S,
                                                              const float* init, int R,
                                                              int BH, long long PN,
                                                              float* h_in) {
  const long long n = (long long)BH * PN;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int bh = (int)(e / PN);
    float hv = init ? init[e] : 0.f;
    h_in[e] = hv;
    for (int r = 0; r < R; ++r) {
      hv = expf(a[(long long)r * BH + bh]) * hv + S[(long long)r * n + e];
      h_in[(long long)(r + 1) * n + e] = hv;
    }
  }
}

}  // namespace

ssd_status_t segment_decay(const void* dt, const float* A, int batch, int T, int H,
                           ssd_dtype_t dtype, float* a, cudaStream_t stream) {
  if (batch * H == 0) return SSD_OK;
  if (dtype == SSD_DT_BF16)
    segment_decay_kernel<true><<<batch * H, 256, 0, stream>>>(dt, A, T, H, a);
  else
    segment_decay_kernel<false><<<batch * H, 256, 0, stream>>>(dt, A, T, H, a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t segment_combine(const float* a, const float* S, const float* init, int R, int batch,
                             int H, int P, int N, float* h_in, cudaStream_t stream) {
  const long long n = (long long)batch * H * P * N;
  if (n == 0) return SSD_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 148 * 16) blocks = 148 * 16;
  segment_combine_kernel<<<(int)blocks, 256, 0, stream>>>(a, S, init, R, batch * H,
                                                         (long long)P * N, h_in);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
