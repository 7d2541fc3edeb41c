// ssd_s6.cu -- the Mamba-1 selective scan (S6) forward: a decay per channel
// and state, the sequential loop of "20.1 상태 공간 모델 (SSM)"
// (sungeuns.github.io), sec. 5 (Selective SSM forward):
//
//     h_t[d,n] = exp(dt_t[d] A[d,n]) h_{t-1}[d,n] + dt_t[d] B_t[n] x_t[d]
//     y_t[d]   = sum_n h_t[d,n] C_t[n] + D[d] x_t[d]
//
// Unlike SSD, the decay differs for every (d, n), so the scan has no matrix
// form: every (t, d, n) takes its own exponential.  The same page calls this
// the step that Mamba-1 runs as a parallel scan over time and Mamba-2
// replaces by SSD block matrix products.
//
// Mapping.  LPC lanes of a warp share one channel d, lane s of the group
// holds states n = s*NS .. s*NS+NS-1 in registers and walks the sequence in
// order (there are batch*Dm*LPC independent lanes, enough to fill the GPU
// without splitting time).  The sequence is taken in blocks of LPC steps.
// Per block a lane loads x and dt of one step of its channel (kPf blocks
// ahead into registers, after an L2 prefetch kL2 blocks ahead: these reads
// are scattered 2- or 4-byte pieces of DRAM rows) and the values are
// broadcast to the group with shuffles.  The B and C rows of a block, which
// every channel needs, are copied into a shared-memory ring with cp.async
// kRing - 1 blocks ahead and read by all warps of the thread block.  The
// output sum over the LPC lanes of a channel is deferred: each lane keeps its
// partial sums of LPC steps and a butterfly reduce-scatter over the group
// leaves lane s with the full sum of step s.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr float kLog2eS6 = 1.4426950408889634f;
constexpr int kPf = 4;  // step blocks of x and dt loaded ahead
constexpr int kL2 = 16; // step blocks of x and dt prefetched into L2 ahead

__device__ __forceinline__ float s6_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ float ld1(const void* p, long long i) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

// NS consecutive elements starting at element i (i a multiple of NS).
template <bool BF16, int NS>
__device__ __forceinline__ void ldv(const void* p, long long i, float (&v)[NS]) {
  if (BF16) {
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p) + i;
    if constexpr (NS % 8 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(q + k);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[k + 2 * j] = __uint_as_float(u[j] << 16);
          v[k + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
      }
    } else if constexpr (NS % 2 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(q + k);
        v[k] = __uint_as_float(w << 16);
        v[k + 1] = __uint_as_float(w & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int k = 0; k < NS; ++k) v[k] = __bfloat162float(q[k]);
    }
  } else {
    const float* q = reinterpret_cast<const float*>(p) + i;
    if constexpr (NS % 4 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 4) {
        const float4 w = *reinterpret_cast<const float4*>(q + k);
        v[k] = w.x;
        v[k + 1] = w.y;
        v[k + 2] = w.z;
        v[k + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < NS; ++k) v[k] = q[k];
    }
  }
}

struct S6Params {
  const void *x, *dt, *B, *C;
  const float *A, *D, *init;
  float *y, *final_states;
  int L, Dm, N;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int K>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}

// NS consecutive elements of a shared-memory row segment.
template <bool BF16, int NS>
__device__ __forceinline__ void lds_v(const uint8_t* p, float (&v)[NS]) {
  if (BF16) {
    if constexpr (NS % 8 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(p + 2 * k);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[k + 2 * j] = __uint_as_float(u[j] << 16);
          v[k + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
      }
    } else if constexpr (NS % 2 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p + 2 * k);
        v[k] = __uint_as_float(w << 16);
        v[k + 1] = __uint_as_float(w & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int k = 0; k < NS; ++k)
        v[k] = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p + 2 * k) << 16);
    }
  } else {
    if constexpr (NS % 4 == 0) {
#pragma unroll
      for (int k = 0; k < NS; k += 4) {
        const float4 w = *reinterpret_cast<const float4*>(p + 4 * k);
        v[k] = w.x;
        v[k + 1] = w.y;
        v[k + 2] = w.z;
        v[k + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < NS; ++k) v[k] = reinterpret_cast<const float*>(p)[k];
    }
  }
}

// Shared memory of a block: a ring of kRing step blocks, each the LPC rows
// of B then the LPC rows of C (N elements each), read by all its warps.
template <int NS, int LPC, bool BF16>
__host__ __device__ constexpr int s6_block_bytes() {
  return 2 * LPC * NS * LPC * (BF16 ? 2 : 4);
}
constexpr int kRing = 3;

// W warps per block; a warp holds 32 / LPC channels.  Grid: (channel
// groups, batch).
template <int NS, int LPC, int W, bool BF16>
__global__ void __launch_bounds__(32 * W) s6_scan_kernel(S6Params p) {
  constexpr int kCh = 32 / LPC;  // channels per warp
  constexpr int kChB = W * kCh;  // channels per block
  constexpr int kEs = BF16 ? 2 : 4;
  constexpr int kN = NS * LPC;   // dstate
  constexpr int kRowBytes = kN * kEs;
  constexpr int kBlk = s6_block_bytes<NS, LPC, BF16>();
  constexpr int kChunks = kBlk / 16;  // 16-byte copies per step block
  static_assert(kRowBytes % 16 == 0, "B/C rows must be whole 16-byte chunks");
  extern __shared__ __align__(16) uint8_t s6_smem[];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int s = lane % LPC;      // state group of this lane
  const int grp = lane / LPC;
  const int b = blockIdx.y;
  const int d = blockIdx.x * kChB + (tid >> 5) * kCh + grp;
  const bool live = d < p.Dm;
  const int dc = live ? d : p.Dm - 1;  // a valid channel for the loads of idle lanes
  const int n0 = s * NS;

  float a2[NS], h[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    a2[k] = live ? p.A[(long long)dc * kN + n0 + k] * kLog2eS6 : 0.f;
    h[k] = (live && p.init) ? p.init[((long long)b * p.Dm + dc) * kN + n0 + k] : 0.f;
  }
  const float Dd = (live && p.D) ? p.D[dc] : 0.f;
  const long long row0 = (long long)b * p.L;
  const int nblk = (p.L + LPC - 1) / LPC;

  // B and C rows of step block `blk` into ring slot blk % kRing (rows past
  // the end repeat the last row: their steps have dt = 0 and no output)
  auto fetch = [&](int blk) {
    if (blk < nblk) {
      uint8_t* dst = s6_smem + (blk % kRing) * kBlk;
#pragma unroll
      for (int c = tid; c < kChunks; c += 32 * W) {
        const int off = c * 16;
        const int half = off / (LPC * kRowBytes);  // 0: B, 1: C
        const int rem = off - half * LPC * kRowBytes;
        const int j = rem / kRowBytes;
        int t = blk * LPC + j;
        t = t < p.L ? t : p.L - 1;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(half ? p.C : p.B) +
                             (row0 + t) * kRowBytes + (rem - j * kRowBytes);
        cp_async16(dst + off, src);
      }
    }
    cp_async_commit();
  };
  // x and dt of step t (0 past the end: the state is then left unchanged,
  // exp(0) = 1 and no input), for lane s of its channel group
  auto xdt = [&](int t, float& xv, float& dv) {
    const bool tv = live && t < p.L;
    xv = tv ? ld1<BF16>(p.x, (row0 + t) * p.Dm + dc) : 0.f;
    dv = tv ? ld1<BF16>(p.dt, (row0 + t) * p.Dm + dc) : 0.f;
  };
  // x and dt come from DRAM: each lane keeps the values of the next kPf
  // step blocks in flight; B and C are staged kRing - 1 blocks ahead
  float xq[kPf], dq[kPf];
#pragma unroll
  for (int q = 0; q < kPf; ++q) xdt(q * LPC + s, xq[q], dq[q]);
#pragma unroll
  for (int q = 0; q < kRing - 1; ++q) fetch(q);

  for (int tq = 0; tq < nblk; tq += kPf) {
#pragma unroll
    for (int q = 0; q < kPf; ++q) {
      const int blk = tq + q;
      if (blk >= nblk) break;
      const int t0 = blk * LPC;
      const float xs = xq[q], ds = dq[q];
      xdt(t0 + kPf * LPC + s, xq[q], dq[q]);
      {
        // x and dt rows of a block kL2 blocks ahead into L2 (one lane per
        // row and tensor; the channel group's values share one sector)
        const int tp = t0 + kL2 * LPC + (tid % LPC);
        if (tid < 2 * LPC && tp < p.L) {
          const void* base = tid < LPC ? p.x : p.dt;
          const uint8_t* a = reinterpret_cast<const uint8_t*>(base) +
                             ((row0 + tp) * p.Dm + (long long)blockIdx.x * kChB) * (BF16 ? 2 : 4);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
      }
      fetch(blk + kRing - 1);
      cp_async_wait<kRing - 1>();
      __syncthreads();
      const uint8_t* sb = s6_smem + (blk % kRing) * kBlk + n0 * kEs;
      float part[LPC];
#pragma unroll
      for (int j = 0; j < LPC; ++j) {
        const float xt = __shfl_sync(0xffffffffu, xs, j, LPC);
        const float dtt = __shfl_sync(0xffffffffu, ds, j, LPC);
        float bv[NS], cv[NS];
        lds_v<BF16, NS>(sb + j * kRowBytes, bv);
        lds_v<BF16, NS>(sb + (LPC + j) * kRowBytes, cv);
        const float u = dtt * xt;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          const float dA = s6_exp2(dtt * a2[k]);
          h[k] = fmaf(dA, h[k], u * bv[k]);
          acc = fmaf(h[k], cv[k], acc);
        }
        part[j] = acc;
      }
      // every thread has read this slot before it is refilled
      __syncthreads();
      // reduce-scatter over the LPC lanes of the channel: after the rounds,
      // lane s holds the sum over the group of part[s]
#pragma unroll
      for (int o = LPC / 2, V = LPC; o >= 1; o >>= 1, V >>= 1) {
        const bool up = (s & o) != 0;
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
          const float send = up ? part[i] : part[i + V / 2];
          const float keep = up ? part[i + V / 2] : part[i];
          part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o, LPC);
        }
      }
      const int ts = t0 + s;
      if (live && ts < p.L) p.y[(row0 + ts) * p.Dm + d] = fmaf(Dd, xs, part[0]);
    }
  }
  cp_async_wait<0>();
  if (live && p.final_states) {
#pragma unroll
    for (int k = 0; k < NS; ++k) p.final_states[((long long)b * p.Dm + d) * kN + n0 + k] = h[k];
  }
}

template <int NS, int LPC, int W>
cudaError_t launch_s6(const S6Params& p, int batch, bool bf16, cudaStream_t st) {
  constexpr int kChB = W * (32 / LPC);
  const dim3 grid((p.Dm + kChB - 1) / kChB, batch);
  if (bf16) {
    constexpr int smem = kRing * s6_block_bytes<NS, LPC, true>();
    auto k = s6_scan_kernel<NS, LPC, W, true>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k<<<grid, 32 * W, smem, st>>>(p);
  } else {
    constexpr int smem = kRing * s6_block_bytes<NS, LPC, false>();
    auto k = s6_scan_kernel<NS, LPC, W, false>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k<<<grid, 32 * W, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

ssd_status_t s6_forward(const void* x, const void* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* init, int batch, int L,
                        int Dm, int N, ssd_dtype_t dtype, float* y, float* final_states,
                        cudaStream_t stream) {
  S6Params p{x, dt, B, C, A, D, init, y, final_states, L, Dm, N};
  const bool bf16 = dtype == SSD_DT_BF16;
  cudaError_t e;
  switch (N) {
    case 16: e = launch_s6<2, 8, 1>(p, batch, bf16, stream); break;
    case 32: e = launch_s6<4, 8, 1>(p, batch, bf16, stream); break;
    case 64: e = launch_s6<4, 16, 2>(p, batch, bf16, stream); break;
    case 128: e = launch_s6<8, 16, 2>(p, batch, bf16, stream); break;
    case 256: e = launch_s6<16, 16, 2>(p, batch, bf16, stream); break;
    default: return SSD_ERR_UNSUPPORTED;
  }
  count_launches(1);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
