// ssd_decode.cu -- single-token state update (decode step).
//
// One iteration of the recurrence applied to a stored state, in place
// ("Transformers are SSMs Review", sec. 1-1: a constant-size state replaces
// the growing KV cache; the update is the loop body of
// "20.1 상태 공간 모델 (SSM)", sec. 5):
//
//   a = exp(dt[b,h] * A[h])
//   state[b,h,p,n] = a * state[b,h,p,n] + dt[b,h] * x[b,h,p] * B[b,g,n]
//   y[b,h,p]       = sum_n C[b,g,n] * state[b,h,p,n] + D[h] * x[b,h,p]
//
// The step is a pure HBM stream: every state element is read once and
// written once (8 bytes per element; the per-row inputs are noise).  One
// 256-thread block per (b, h); each thread owns a 16-byte column slice of N
// (float4) and walks rows p, so a warp reads whole 128-byte lines and the y
// reduction over n is a segmented shuffle inside the warp.  All of a
// thread's row loads are issued before any arithmetic to keep enough bytes
// in flight.
#include <cuda_bf16.h>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kDecThreads = 256;

template <typename Tin>
__device__ __forceinline__ float4 ld4_in(const Tin* p);
template <>
__device__ __forceinline__ float4 ld4_in<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 ld4_in<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xffff0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xffff0000u);
  return r;
}

// LANES = threads per state row (N/4 columns of float4, capped at 32);
// VEC = float4 per thread per row (N/4 / LANES); ROWS = rows per thread
// batch issued together.
template <typename Tin, int LANES, int VEC, int ROWS>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(
    float* __restrict__ state, const Tin* __restrict__ x, const Tin* __restrict__ dt,
    const float* __restrict__ A, const Tin* __restrict__ B, const Tin* __restrict__ C,
    const float* __restrict__ D, int H, int P, int G, float* __restrict__ y) {
  constexpr int N = LANES * VEC * 4;
  constexpr int kRowsPerPass = kDecThreads / LANES;
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int g = (int)((long long)h * G / H);
  const int lane_in_row = threadIdx.x % LANES;
  const int row0 = threadIdx.x / LANES;
  const float dtv = ld_in(dt + bh);
  const float a = expf(dtv * A[h]);
  const float Dh = D ? D[h] : 0.f;
  float4 bv[VEC], cv[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    const int n = (v * LANES + lane_in_row) * 4;
    bv[v] = ld4_in<Tin>(B + ((long long)b * G + g) * N + n);
    cv[v] = ld4_in<Tin>(C + ((long long)b * G + g) * N + n);
  }
  float* st = state + (long long)bh * P * N;
  const Tin* xr = x + (long long)bh * P;
  for (int p0 = row0; p0 < P; p0 += kRowsPerPass * ROWS) {
    float4 s[ROWS][VEC];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int p = p0 + r * kRowsPerPass;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        const int n = (v * LANES + lane_in_row) * 4;
        s[r][v] = p < P ? __ldcs(reinterpret_cast<const float4*>(st + (long long)p * N + n))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int p = p0 + r * kRowsPerPass;
      const float xp = p < P ? ld_in(xr + p) : 0.f;
      const float u = dtv * xp;
      float part = 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float4 e = s[r][v];
        e.x = a * e.x + u * bv[v].x;
        e.y = a * e.y + u * bv[v].y;
        e.z = a * e.z + u * bv[v].z;
        e.w = a * e.w + u * bv[v].w;
        part += cv[v].x * e.x + cv[v].y * e.y + cv[v].z * e.z + cv[v].w * e.w;
        const int n = (v * LANES + lane_in_row) * 4;
        if (p < P) __stcs(reinterpret_cast<float4*>(st + (long long)p * N + n), e);
      }
#pragma unroll
      for (int o = LANES / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane_in_row == 0 && p < P) y[(long long)bh * P + p] = part + Dh * xp;
    }
  }
}

template <typename Tin, int LANES, int VEC>
cudaError_t launch_decode(float* state, const void* x, const void* dt, const float* A,
                          const void* B, const void* C, const float* D, int batch, int H, int P,
                          int G, float* y, cudaStream_t stream) {
  const long long blocks = (long long)batch * H;
  if (blocks == 0) return cudaSuccess;
  decode_kernel<Tin, LANES, VEC, 8><<<(unsigned)blocks, kDecThreads, 0, stream>>>(
      state, static_cast<const Tin*>(x), static_cast<const Tin*>(dt), A,
      static_cast<const Tin*>(B), static_cast<const Tin*>(C), D, H, P, G, y);
  count_launches(1);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t decode_dispatch(float* state, const void* x, const void* dt, const float* A,
                            const void* B, const void* C, const float* D, int batch, int H,
                            int P, int N, int G, float* y, cudaStream_t s) {
  switch (N) {
    case 16: return launch_decode<Tin, 4, 1>(state, x, dt, A, B, C, D, batch, H, P, G, y, s);
    case 32: return launch_decode<Tin, 8, 1>(state, x, dt, A, B, C, D, batch, H, P, G, y, s);
    case 64: return launch_decode<Tin, 16, 1>(state, x, dt, A, B, C, D, batch, H, P, G, y, s);
    case 128: return launch_decode<Tin, 32, 1>(state, x, dt, A, B, C, D, batch, H, P, G, y, s);
    case 256: return launch_decode<Tin, 32, 2>(state, x, dt, A, B, C, D, batch, H, P, G, y, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

ssd_status_t decode_step(float* state, const void* x, const void* dt, const float* A,
                         const void* B, const void* C, const float* D, int batch, int H, int P,
                         int N, int G, ssd_dtype_t dtype, float* y, cudaStream_t stream) {
  cudaError_t e = dtype == SSD_DT_BF16
                      ? decode_dispatch<__nv_bfloat16>(state, x, dt, A, B, C, D, batch, H, P, N,
                                                       G, y, stream)
                      : decode_dispatch<float>(state, x, dt, A, B, C, D, batch, H, P, N, G, y,
                                               stream);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
