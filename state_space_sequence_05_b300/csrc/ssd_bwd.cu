// ssd_bwd.cu -- backward of the SSD layer forward: the gradients of a loss L
// with respect to x, dt, A, B, C, D and the initial state, given dL/dy and
// dL/dfinal.  The reverse-mode derivative of the recurrence
//
//     h_t = a_t h_{t-1} + dt_t x_t B_t^T,  a_t = exp(dt_t A),  y_t = h_t C_t + D x_t
//
// ("20.1 상태 공간 모델 (SSM)", sec. 1 and the sec. 5 loop; scalar A per head
// and B, C shared by a group, "Transformers are SSMs Review", sec. 3-2) runs
// the adjoint G_t = dL/dh_t backwards in time:
//
//     G_t = dy_t C_t^T + a_{t+1} G_{t+1}   (G_{T-1} starts from dL/dfinal)
//     dx_t = dt_t G_t B_t + D dy_t,  dB_t = dt_t G_t^T x_t,  dC_t = h_t^T dy_t,
//     ddt_t = <G_t, A a_t h_{t-1} + x_t B_t^T>,  dA = sum_t dt_t a_t <G_t, h_{t-1}>,
//     dD = sum_t <dy_t, x_t>,  dinit = a_0 G_0.
//
// Design: the rows p of the state never mix (h_t[p,:] and G_t[p,:] evolve on
// their own), so the work is cut into blocks of (batch row, head, slice of
// kRows state rows), the slice's state and adjoint in shared memory.  Sums
// over p (dB, dC, ddt, dA, dD) add up the slices with atomics (the entry
// point zeroes them first).  The states h_t are needed in reverse
// order: a first forward sweep stores every kCk-th state in the workspace;
// then, chunk by chunk from the end, the chunk's kCk states are recomputed
// from its checkpoint into the workspace and the adjoint walks the chunk
// backwards.  Sums over a row of the state go to warps, sums over a column to
// threads.  All arithmetic is fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kCk = 64;   // steps between stored states
constexpr int kRows = 8;  // state rows per block

struct BwdParams {
  const void *x, *dt, *B, *C;
  const float *A, *D, *init, *dy, *dfinal;
  float *dx, *ddt, *dA, *dB, *dC, *dD, *dinit;
  float* ws;  // per (b, h, slice): (nck + 1) stored states, then kCk chunk states
  int T, H, P, N, G, nck, nslice;
};

template <bool BF16>
__device__ __forceinline__ float ldin(const void* p, long long i) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <bool BF16>
__global__ void __launch_bounds__(kBwdThreads) ssd_bwd_kernel(BwdParams p) {
  const int bh = blockIdx.x / p.nslice;
  const int slice = blockIdx.x % p.nslice;
  const int b = bh / p.H, h = bh % p.H;
  const int g = (int)((long long)h * p.G / p.H);
  const int N = p.N, H = p.H, G = p.G, Pf = p.P;
  const int p0 = slice * kRows;                 // first state row of this block
  const int P = min(kRows, Pf - p0);            // rows of this block
  const int PN = P * N;                         // state elements of this block
  const long long soff = ((long long)bh * Pf + p0) * N;  // its offset in a [b, H, P, N] state
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ float bwd_smem[];
  float* hsm = bwd_smem;     // [PN] running state
  float* Gsm = hsm + PN;     // [PN] adjoint
  float* xs = Gsm + PN;      // [P]  x_t
  float* dys = xs + P;       // [P]  dy_t
  float* Bs = dys + P;       // [N]  B_t
  float* Cs = Bs + N;        // [N]  C_t
  float* red = Cs + N;       // [2 * kBwdWarps] block-sum partials

  const float Ah = p.A[h];
  const float Dh = p.D ? p.D[h] : 0.f;
  const long long tok0 = (long long)b * p.T;
  float* ck = p.ws + (long long)blockIdx.x * (p.nck + 1 + kCk) * (kRows * N);  // stored states
  float* hs = ck + (long long)(p.nck + 1) * PN;                                // one chunk's states

  // inputs of step t into shared memory (callers synchronise around it)
  auto load_step = [&](int t, bool backward) {
    const long long bt = tok0 + t;
    for (int i = tid; i < P; i += kBwdThreads) {
      xs[i] = ldin<BF16>(p.x, (bt * H + h) * Pf + p0 + i);
      if (backward) dys[i] = p.dy[(bt * H + h) * Pf + p0 + i];
    }
    for (int i = tid; i < N; i += kBwdThreads) {
      Bs[i] = ldin<BF16>(p.B, (bt * G + g) * N + i);
      if (backward) Cs[i] = ldin<BF16>(p.C, (bt * G + g) * N + i);
    }
  };
  // hsm <- a_t hsm + dt_t x_t B_t^T (each thread updates the elements it owns)
  auto step_forward = [&](int t) {
    const float dtt = ldin<BF16>(p.dt, (tok0 + t) * H + h);
    const float a = expf(dtt * Ah);
    __syncthreads();
    load_step(t, false);
    __syncthreads();
    for (int e = tid; e < PN; e += kBwdThreads) {
      const int pp = e / N, n = e - pp * N;
      hsm[e] = a * hsm[e] + dtt * xs[pp] * Bs[n];
    }
  };

  // 1. forward sweep, storing the state before every kCk-th step
  for (int e = tid; e < PN; e += kBwdThreads) {
    const float v = p.init ? p.init[soff + e] : 0.f;
    hsm[e] = v;
    ck[e] = v;
  }
  for (int t = 0; t < p.T; ++t) {
    step_forward(t);
    if ((t + 1) % kCk == 0 && t + 1 < p.T)
      for (int e = tid; e < PN; e += kBwdThreads) ck[(long long)((t + 1) / kCk) * PN + e] = hsm[e];
  }

  // 2. the adjoint, chunk by chunk from the end
  for (int e = tid; e < PN; e += kBwdThreads)
    Gsm[e] = p.dfinal ? p.dfinal[soff + e] : 0.f;
  float dA_acc = 0.f, dD_acc = 0.f;  // thread 0's running sums
  for (int c = p.nck - 1; c >= 0; --c) {
    const int t0 = c * kCk;
    const int t1 = min(p.T, t0 + kCk);
    // this chunk's states h_t0 .. h_{t1-1}, from the state before t0
    for (int e = tid; e < PN; e += kBwdThreads) hsm[e] = ck[(long long)c * PN + e];
    for (int t = t0; t < t1; ++t) {
      step_forward(t);
      for (int e = tid; e < PN; e += kBwdThreads) hs[(long long)(t - t0) * PN + e] = hsm[e];
    }
    for (int t = t1 - 1; t >= t0; --t) {
      const long long bt = tok0 + t;
      const float dtt = ldin<BF16>(p.dt, bt * H + h);
      const float a = expf(dtt * Ah);
      const float* ht = hs + (long long)(t - t0) * PN;
      const float* hp = t > t0 ? hs + (long long)(t - t0 - 1) * PN : ck + (long long)c * PN;
      __syncthreads();  // the previous step is done with the shared inputs and sums
      load_step(t, true);
      __syncthreads();
      // G_t = dy_t C_t^T + (the decayed adjoint of the later steps)
      float s_h = 0.f, s_xb = 0.f;
      for (int e = tid; e < PN; e += kBwdThreads) {
        const int pp = e / N, n = e - pp * N;
        const float gv = Gsm[e] + dys[pp] * Cs[n];
        Gsm[e] = gv;
        s_h += gv * hp[e];
        s_xb += gv * xs[pp] * Bs[n];
      }
      s_h = warp_sum(s_h);
      s_xb = warp_sum(s_xb);
      if (lane == 0) {
        red[warp] = s_h;
        red[kBwdWarps + warp] = s_xb;
      }
      __syncthreads();  // G_t and the partial sums are complete
      // dx_t[p] = dt_t sum_n G_t[p,n] B_t[n] + D dy_t[p]: a warp per row
      for (int pp = warp; pp < P; pp += kBwdWarps) {
        float acc = 0.f;
        for (int n = lane; n < N; n += 32) acc += Gsm[pp * N + n] * Bs[n];
        acc = warp_sum(acc);
        if (lane == 0) p.dx[(bt * H + h) * Pf + p0 + pp] = dtt * acc + Dh * dys[pp];
      }
      // dB_t[n] += dt_t sum_p G_t[p,n] x_t[p], dC_t[n] += sum_p dy_t[p] h_t[p,n]
      for (int n = tid; n < N; n += kBwdThreads) {
        float gb = 0.f, gc = 0.f;
        for (int pp = 0; pp < P; ++pp) {
          gb += Gsm[pp * N + n] * xs[pp];
          gc += dys[pp] * ht[pp * N + n];
        }
        atomicAdd(p.dB + (bt * G + g) * N + n, dtt * gb);
        atomicAdd(p.dC + (bt * G + g) * N + n, gc);
      }
      if (tid == 0) {
        float sh = 0.f, sxb = 0.f;
        for (int w = 0; w < kBwdWarps; ++w) {
          sh += red[w];
          sxb += red[kBwdWarps + w];
        }
        atomicAdd(p.ddt + bt * H + h, Ah * a * sh + sxb);
        dA_acc += dtt * a * sh;
        float xd = 0.f;
        for (int pp = 0; pp < P; ++pp) xd += dys[pp] * xs[pp];
        dD_acc += xd;
      }
      __syncthreads();  // every reader of G_t is done
      // dL/dh_{t-1} through the recurrence
      for (int e = tid; e < PN; e += kBwdThreads) Gsm[e] *= a;
    }
  }
  if (p.dinit)
    for (int e = tid; e < PN; e += kBwdThreads) p.dinit[soff + e] = Gsm[e];
  if (tid == 0) {
    atomicAdd(p.dA + h, dA_acc);
    if (p.dD) atomicAdd(p.dD + h, dD_acc);
  }
}

// shared memory of a block holding `rows` state rows (the kernel's layout:
// state, adjoint, x, dy, B, C, block-sum partials)
size_t smem_bytes(int rows, int N) {
  return sizeof(float) * ((size_t)2 * rows * N + 2 * rows + 2 * N + 2 * kBwdWarps);
}

}  // namespace

size_t bwd_workspace_bytes(int batch, int T, int H, int P, int N) {
  const long long nck = ((long long)T + kCk - 1) / kCk;
  const long long nslice = (P + kRows - 1) / kRows;
  const size_t steps = sizeof(float) * (size_t)batch * H * nslice * (size_t)(nck + 1 + kCk) * kRows * N;
  // either backward may run a supported shape (the chunked one needs 16-byte
  // aligned state arguments)
  if (!bwd_chunked_supported(P, N)) return steps;
  const size_t chunked = bwd_chunked_workspace_bytes(batch, T, H, P, N);
  return chunked > steps ? chunked : steps;
}

ssd_status_t bwd(const BwdArgs& a) {
  BwdParams p;
  p.x = a.x;
  p.dt = a.dt;
  p.B = a.B;
  p.C = a.C;
  p.A = a.A;
  p.D = a.D;
  p.init = a.init;
  p.dy = a.dy;
  p.dfinal = a.dfinal;
  p.dx = a.dx;
  p.ddt = a.ddt;
  p.dA = a.dA;
  p.dB = a.dB;
  p.dC = a.dC;
  p.dD = a.dD;
  p.dinit = a.dinit;
  p.ws = static_cast<float*>(a.ws);
  p.T = a.seqlen;
  p.H = a.H;
  p.P = a.P;
  p.N = a.N;
  p.G = a.G;
  p.nck = (a.seqlen + kCk - 1) / kCk;
  p.nslice = (a.P + kRows - 1) / kRows;
  // the chunked path zeroes the accumulated gradients itself
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (a.seqlen > 0 && bwd_chunked_supported(a.P, a.N) && a16(a.init) && a16(a.dfinal) &&
      a16(a.dinit))
    return bwd_chunked(a);
  if (bwd_zero_grads(a) != cudaSuccess) return SSD_ERR_CUDA;
  if (a.seqlen == 0) {
    // no steps: dinit = dL/dfinal
    if (a.dinit) {
      const size_t n = sizeof(float) * (size_t)a.batch * a.H * a.P * a.N;
      const cudaError_t e = a.dfinal ? cudaMemcpyAsync(a.dinit, a.dfinal, n,
                                                       cudaMemcpyDeviceToDevice, a.stream)
                                     : cudaMemsetAsync(a.dinit, 0, n, a.stream);
      if (e != cudaSuccess) return SSD_ERR_CUDA;
    }
    return SSD_OK;
  }
  const size_t smem = smem_bytes(a.P < kRows ? a.P : kRows, a.N);
  auto k = a.dtype == SSD_DT_BF16 ? ssd_bwd_kernel<true> : ssd_bwd_kernel<false>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return SSD_ERR_CUDA;
  k<<<a.batch * a.H * p.nslice, kBwdThreads, smem, a.stream>>>(p);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

cudaError_t bwd_zero_grads(const BwdArgs& a) {
  const long long ntok = (long long)a.batch * a.seqlen;
  cudaError_t e = cudaMemsetAsync(a.dA, 0, sizeof(float) * a.H, a.stream);
  if (e == cudaSuccess && ntok > 0) e = cudaMemsetAsync(a.ddt, 0, sizeof(float) * ntok * a.H, a.stream);
  if (e == cudaSuccess && a.dD) e = cudaMemsetAsync(a.dD, 0, sizeof(float) * a.H, a.stream);
  if (e == cudaSuccess && ntok > 0)
    e = cudaMemsetAsync(a.dB, 0, sizeof(float) * ntok * a.G * a.N, a.stream);
  if (e == cudaSuccess && ntok > 0)
    e = cudaMemsetAsync(a.dC, 0, sizeof(float) * ntok * a.G * a.N, a.stream);
  return e;
}

}  // namespace ssd
