// ssd_bwd_chunked.cu -- chunked backward of the SSD layer forward for
// headdim <= 64 and dstate <= 128 (batch mode): the gradients of a loss L
// with respect to x, dt, A, B, C, D and the initial state, given dL/dy and
// dL/dfinal, through the forward's chunked form ("Transformers are SSMs
// Review", sec. 3-2 (4)) instead of a walk over every step.
//
// Forward, per chunk c of 64 tokens (cum_i = sum_{k<=i} dt_k A chunk-local,
// L_ij = exp(cum_i - cum_j) for j <= i, G_ij = C_i . B_j, M_ij = G_ij L_ij dt_j,
// w_j = exp(cum_last - cum_j) dt_j, H_c the state entering the chunk):
//
//   y_i      = sum_j M_ij x_j + exp(cum_i) H_c C_i + D x_i
//   H_{c+1}  = exp(cum_last) H_c + sum_j w_j x_j B_j^T
//
// Backward.  The adjoint of the state leaving chunk c, dH_{c+1}, runs
// backwards over chunks like the forward state runs forwards:
//
//   dH_c = exp(cum_last) dH_{c+1} + sum_i exp(cum_i) dy_i C_i^T,
//
// starting from dL/dfinal after the last chunk; dinit = dH_0.  Within a
// chunk, with dS_ij = dy_i . x_j and dG_ij = dS_ij L_ij dt_j:
//
//   dx_j  = sum_i M_ij dy_i + w_j dH_{c+1} B_j + D dy_j
//   dC_i  = sum_j dG_ij B_j + exp(cum_i) H_c^T dy_i
//   dB_j  = sum_i dG_ij C_i + w_j dH_{c+1}^T x_j
//   dD    = sum_i dy_i . x_i
//
// and the decay terms through dcum_k = dL/dcum_k (chunk-local):
//
//   dcum_i += sum_j dS_ij M_ij + exp(cum_i) C_i . (H_c^T dy_i)      (row i)
//   dcum_j -= sum_i dS_ij M_ij + w_j x_j . (dH_{c+1} B_j)           (column j)
//   dcum_last += exp(cum_last) <dH_{c+1}, H_c> + sum_j w_j x_j . (dH_{c+1} B_j)
//   ddt_j = sum_i dS_ij G_ij L_ij + exp(cum_last - cum_j) x_j . (dH_{c+1} B_j)
//           + A sum_{k>=j} dcum_k
//   dA    = sum_j dt_j sum_{k>=j} dcum_k          (over every chunk)
//
// Kernels (fp32 accumulation; the products on tensor cores take fp32
// operands as bf16 hi/lo pairs, hi = rn(v), lo = rn(v - hi)):
//   bwd_outer_kernel<F>  per (chunk, group, slice of up to 10 of the group's
//                        heads): the chunk states sum_j w_j x_j B_j^T and
//                        exp(cum_last), warp MMAs;
//   bwd_outer_kernel<R>  the same for sum_i exp(cum_i) dy_i C_i^T;
//   bwd_pass_kernel      per (row, head, state element): the states entering
//                        each chunk (forwards) / the adjoints leaving each
//                        chunk (backwards), in place; dinit;
//   bwd_tab_kernel       per (chunk, head): the forward and adjoint weights
//                        and the chunk decay; it also zeroes the gradients
//                        the other kernels accumulate;
//   bwd_scan_kernel      per (head, batch row, direction, half of headdim):
//                        the states entering and the adjoints leaving every
//                        chunk (tcgen05 chunk sums, operands by TMA), written
//                        as bf16 hi/lo pairs;
//   bwd_grad_tc_kernel   per (chunk, group, slice of up to 10 heads), bf16
//                        inputs with headdim and dstate multiples of 8:
//                        every gradient above on tcgen05 MMAs (M = 64 per
//                        head), dB and dC transposed (M = 128) and summed
//                        over the slice in tensor memory;
//   bwd_grad_kernel      the same on CUDA cores for fp32 inputs and other
//                        shapes, dB and dC summed over the slice in
//                        registers.
// dB, dC, dA and dD are added with atomics into zeroed buffers: on the
// tensor-core path the weight-table kernel clears them (and ddt) first, on
// the CUDA-core path memsets do.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "ssd.h"
#include "ssd_internal.h"
#include "ssd_tc_host.h"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace ssd {
namespace {

constexpr int kQb = 64;     // chunk length
constexpr int kThr = 256;   // threads per block
constexpr int kPmax = 64;   // headdim of this path, at most
constexpr int kNmax = 128;  // dstate of this path, at most
constexpr int kNT = 32;     // dstate columns per tile of H / dH in the gradient kernel

struct BP {
  const void *x, *dt, *B, *C;
  const float *A, *D, *init, *dy, *dfinal;
  float *dx, *ddt, *dA, *dB, *dC, *dD, *dinit;
  int32_t* status;  // SSD_ERR_TIMEOUT when a device wait runs out (may be null)
  unsigned wait_polls;  // bound on every mbarrier wait of the tcgen05 kernels (polls)
  int hold;             // test hook: 1 / 2 hold back one MMA completion (gradients / scans)
  float* st;   // [chunks][H][P N]: chunk states, then the states entering each chunk
  float* ad;   // [chunks][H][P N]: local adjoint sums, then the adjoints leaving each chunk
  // tensor-core path: the same two buffers hold the transposed states as bf16
  // hi/lo pairs, [chunks][H][N][P] each (st = sth | stl, ad = adh | adl)
  __nv_bfloat16 *sth, *stl, *adh, *adl;
  float* dec;  // [chunks][H]: exp(cum_last)
  float* tab;  // [chunks][H][144] (tensor-core path): forward weights, adjoint weights, decay
  int T, H, P, N, G, nc;  // nc: chunks per batch row
  int vec;  // rows of x, dy, B, C move as 16-byte vectors (headdim, dstate multiples of 8)
};

template <bool BF16>
__device__ __forceinline__ float ldin(const void* p, long long i) {
  if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return reinterpret_cast<const float*>(p)[i];
}

// Where chunk `c` (global index) lies: batch row, first token, valid rows.
struct Chunk {
  int b, t0, len;
  long long tok0;  // global index of its first token
};
__device__ __forceinline__ Chunk chunk_of(const BP& p, int c) {
  Chunk k;
  k.b = c / p.nc;
  k.t0 = (c % p.nc) * kQb;
  k.len = min(kQb, p.T - k.t0);
  k.tok0 = (long long)k.b * p.T + k.t0;
  return k;
}

// cum[j] = sum_{k<=j} dt_k A (j < 64; dt = 0 past the valid rows) and dts[j]
// = dt_j, by threads 0..63 (two warp scans).  Ends with a block barrier.
template <bool BF16>
__device__ __forceinline__ void chunk_cum(const BP& p, const Chunk& k, int h, float Ah, float* cum,
                                          float* dts, float* wsum) {
  const int t = threadIdx.x;
  if (t < kQb) {
    const float d = t < k.len ? ldin<BF16>(p.dt, (k.tok0 + t) * p.H + h) : 0.f;
    float v = d * Ah;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if ((t & 31) >= o) v += u;
    }
    if ((t & 31) == 31) wsum[t >> 5] = v;
    cum[t] = v;
    dts[t] = d;
  }
  __syncthreads();
  if (t >= 32 && t < kQb) cum[t] += wsum[0];
  __syncthreads();
}

// ---------------------------------------------------------------- warp MMA
// Operands of the tensor-core products are fp32 values split into bf16 hi =
// rn(v) and lo = rn(v - hi) (|v - hi - lo| <= 2^-18 |v|); a product of two
// split operands is taken as hi.hi + hi.lo + lo.hi, of a split operand and an
// exact bf16 one as hi.b + lo.b, both accumulated in fp32.
__device__ __forceinline__ void split_rn(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// D (16 x 8, fp32) += A (16 x 16, bf16, row-major fragment) B (16 x 8, bf16)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kAP = kQb + 8;    // pitch (bf16) of the 64 x 64 tiles
constexpr int kBP = kNmax + 8;  // pitch (bf16) of the 64 x 128 tiles
constexpr size_t kT64 = sizeof(__nv_bfloat16) * kQb * kAP;
constexpr size_t kT128 = sizeof(__nv_bfloat16) * kQb * kBP;

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

// Per-lane row/column offsets of the four 8 x 8 matrices of an ldmatrix.x4:
// pattern X for a left operand stored [m][k] and a right operand stored
// [k][n]; pattern Y for a left operand stored [k][m] and a right operand
// stored [n][k].
struct LaneOff {
  int rx, cx, ry, cy;
};
__device__ __forceinline__ LaneOff lane_off(int lane) {
  LaneOff o;
  o.rx = (lane & 7) + ((lane >> 3) & 1) * 8;
  o.cx = (lane >> 4) * 8;
  o.ry = (lane & 7) + (lane >> 4) * 8;
  o.cy = ((lane >> 3) & 1) * 8;
  return o;
}

// acc[t] (16 x 8, t < NT) += A (16 x K) B (K x 8 NT) for k in [kb, ke) (steps
// of 16): A's rows m0.., stored [m][k] (TA false) or [k][m]; B's columns
// n0.., stored [n][k] (TB false) or [k][n].  ALO / BLO: the operand is a
// hi/lo pair (lo at al / bl), else exact in bf16; the hi.hi products go to
// acc, the hi.lo and lo.hi ones to accl (which may be acc).  Per k-step the
// fragments are loaded first and the MMAs issued pass by pass, so that two
// MMAs into one accumulator are NT apart.  Shared addresses in bytes.
template <int NT, int PA, bool TA, bool ALO, int PB, bool TB, bool BLO>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], float (&accl)[NT][4], uint32_t ah_s,
                                         uint32_t al_s, int m0, uint32_t bh_s, uint32_t bl_s,
                                         int n0, int kb, int ke, const LaneOff& o) {
#pragma unroll 1
  for (int k0 = kb; k0 < ke; k0 += 16) {
    const uint32_t aoff = TA ? 2u * ((k0 + o.ry) * PA + m0 + o.cy) : 2u * ((m0 + o.rx) * PA + k0 + o.cx);
    uint32_t ah[4], al[4], bh[NT / 2][4], bl[NT / 2][4];
    if (TA) {
      ldsm4t(ah, ah_s + aoff);
      if (ALO) ldsm4t(al, al_s + aoff);
    } else {
      ldsm4(ah, ah_s + aoff);
      if (ALO) ldsm4(al, al_s + aoff);
    }
#pragma unroll
    for (int u = 0; u < NT / 2; ++u) {
      const int nb = n0 + 16 * u;
      const uint32_t boff = TB ? 2u * ((k0 + o.rx) * PB + nb + o.cx) : 2u * ((nb + o.ry) * PB + k0 + o.cy);
      if (TB) {
        ldsm4t(bh[u], bh_s + boff);
        if (BLO) ldsm4t(bl[u], bl_s + boff);
      } else {
        ldsm4(bh[u], bh_s + boff);
        if (BLO) ldsm4(bl[u], bl_s + boff);
      }
    }
#pragma unroll
    for (int u = 0; u < NT / 2; ++u) {
      mma16816(acc[2 * u], ah, bh[u][0], bh[u][1]);
      mma16816(acc[2 * u + 1], ah, bh[u][2], bh[u][3]);
    }
    if (ALO) {
#pragma unroll
      for (int u = 0; u < NT / 2; ++u) {
        mma16816(accl[2 * u], al, bh[u][0], bh[u][1]);
        mma16816(accl[2 * u + 1], al, bh[u][2], bh[u][3]);
      }
    }
    if (BLO) {
#pragma unroll
      for (int u = 0; u < NT / 2; ++u) {
        mma16816(accl[2 * u], ah, bl[u][0], bl[u][1]);
        mma16816(accl[2 * u + 1], ah, bl[u][2], bl[u][3]);
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
}

__device__ __forceinline__ uint32_t pack_bf2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// four fp32 values -> hi/lo bf16 quadruples (8 bytes each) at dh / dl
__device__ __forceinline__ void store_split4(__nv_bfloat16* dh, __nv_bfloat16* dl, float4 v) {
  __nv_bfloat16 h0, h1, h2, h3, l0, l1, l2, l3;
  split_rn(v.x, h0, l0);
  split_rn(v.y, h1, l1);
  split_rn(v.z, h2, l2);
  split_rn(v.w, h3, l3);
  *reinterpret_cast<uint2*>(dh) = make_uint2(pack_bf2(h0, h1), pack_bf2(h2, h3));
  *reinterpret_cast<uint2*>(dl) = make_uint2(pack_bf2(l0, l1), pack_bf2(l2, l3));
}

// ---------------------------------------------------------------- outer sums
// MODE 0: out = sum_j w_j x_j B_j^T, w_j = exp(cum_last - cum_j) dt_j, into p.st,
//         and exp(cum_last) into p.dec.
// MODE 1: out = sum_i exp(cum_i) dy_i C_i^T into p.ad.
// One block per (chunk, group, slice of up to kHS heads of the group): V (64
// tokens x N) = the group's B or C rows, staged once; per head U (64 tokens x
// P) = the weighted rows, and out = U^T V on the tensor cores (transposing
// loads), warp w taking rows 16 (w % 4).. and columns 64 (w / 4)...  With
// p.vec the rows move as 16-byte vectors: the next head's U rows are copied
// asynchronously into a staging buffer (and its dt loaded) while the current
// head's product runs.
constexpr int kHS = 10;  // heads of a group per block (outer sums and gradients); 80 heads make 8 slices

constexpr size_t kStage = sizeof(float) * kQb * kPmax;  // raw U rows of one head

template <bool BF16>
constexpr size_t outer_smem() {
  return 2 * kT64 + (BF16 ? 1 : 2) * kT128 + kStage + sizeof(float) * kQb;
}

template <bool BF16, int MODE>
__global__ void __launch_bounds__(kThr, 3) bwd_outer_kernel(BP p) {
  extern __shared__ __align__(16) unsigned char osm_raw[];
  __nv_bfloat16* Uh = reinterpret_cast<__nv_bfloat16*>(osm_raw);  // [64 j][72]: hi
  __nv_bfloat16* Ul = Uh + kQb * kAP;                              // lo
  __nv_bfloat16* Vh = Ul + kQb * kAP;                              // [64 j][136]: hi (bf16: exact)
  __nv_bfloat16* Vl = Vh + kQb * kBP;                              // lo (fp32 inputs only)
  unsigned char* stg = reinterpret_cast<unsigned char*>(Vh + (BF16 ? 1 : 2) * kQb * kBP);
  // stg: the next head's U rows as loaded, [64 j][P] (x: input dtype, dy: fp32)
  float* sc = reinterpret_cast<float*>(stg + kStage);  // [64] row weights
  const int c = blockIdx.x, g = blockIdx.y;
  const int hpg = p.H / p.G;
  const int hb = g * hpg + blockIdx.z * kHS;
  const int nh = min(kHS, hpg - blockIdx.z * kHS);
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const Chunk k = chunk_of(p, c);
  const int P = p.P, N = p.N, len = k.len;
  const void* usrc = MODE == 0 ? p.x : static_cast<const void*>(p.dy);
  const void* vsrc = MODE == 0 ? p.B : p.C;
  constexpr int kUS = kQb * kPmax / 4 / kThr;  // 4
  constexpr int kVS = kQb * kNmax / 4 / kThr;  // 8
  (void)kUS;

  // U rows of head h into the staging buffer, 16 bytes per copy (zero past
  // the valid rows); completes at the next cp.async wait
  constexpr bool kUB = MODE == 0 && BF16;  // U rows in bf16
  constexpr int kUE = kUB ? 8 : 4;         // elements per 16 bytes
  constexpr int kUC = kQb * kPmax / kUE / kThr;
  const auto stage_u = [&](int h) {
#pragma unroll
    for (int r = 0; r < kUC; ++r) {
      const int e = t + kThr * r, j = e / (kPmax / kUE), q = (e % (kPmax / kUE)) * kUE;
      const bool ok = j < len && q < P;
      const long long i = ((k.tok0 + (ok ? j : 0)) * p.H + h) * P + (ok ? q : 0);
      const void* src = kUB ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(usrc) + i)
                            : static_cast<const void*>(static_cast<const float*>(usrc) + i);
      tc::cp_async16_zfill(stg + 16 * e, src, ok);
    }
    tc::cp_async_commit();
  };
  // warp 0: dt of head h (rows 2 lane, 2 lane + 1) and then the row weights
  float d0 = 0.f, d1 = 0.f;
  const auto load_dt = [&](int h) {
    const int j0 = 2 * lane, j1 = j0 + 1;
    d0 = j0 < len ? ldin<BF16>(p.dt, (k.tok0 + j0) * p.H + h) : 0.f;
    d1 = j1 < len ? ldin<BF16>(p.dt, (k.tok0 + j1) * p.H + h) : 0.f;
  };
  const auto weights = [&](int h) {
    const float Ah = p.A[h];
    const float a1 = d1 * Ah;
    float s = d0 * Ah + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    const float cm1 = s, cm0 = s - a1;
    const float lst = __shfl_sync(0xffffffffu, ((len - 1) & 1) ? cm1 : cm0, (len - 1) >> 1);
    if (MODE == 0) {
      sc[2 * lane] = expf(lst - cm0) * d0;
      sc[2 * lane + 1] = expf(lst - cm1) * d1;
      if (lane == 0) p.dec[(long long)c * p.H + h] = expf(lst);
    } else {
      sc[2 * lane] = expf(cm0);
      sc[2 * lane + 1] = expf(cm1);
    }
  };

  // ---- V once (zero past the valid rows and dstate)
  if (p.vec) {
    uint2 vb[kVS];
    float4 vf[kVS];
#pragma unroll
    for (int r = 0; r < kVS; ++r) {
      const int e4 = t + kThr * r, j = e4 >> 5, n = (e4 & 31) * 4;
      const bool ok = j < len && n < N;
      const long long i = ((k.tok0 + j) * p.G + g) * N + n;
      if (BF16)
        vb[r] = ok ? *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(vsrc) + i)
                   : make_uint2(0, 0);
      else
        vf[r] = ok ? *reinterpret_cast<const float4*>(static_cast<const float*>(vsrc) + i)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_u(hb);
    if (w == 0) load_dt(hb);
#pragma unroll
    for (int r = 0; r < kVS; ++r) {
      const int e4 = t + kThr * r, j = e4 >> 5, n = (e4 & 31) * 4;
      if (BF16)
        *reinterpret_cast<uint2*>(Vh + j * kBP + n) = vb[r];
      else
        store_split4(Vh + j * kBP + n, Vl + j * kBP + n, vf[r]);
    }
  } else {
    if (w == 0) load_dt(hb);
    for (int e = t; e < kQb * kNmax; e += kThr) {
      const int j = e / kNmax, n = e % kNmax;
      const float v = (j < len && n < N) ? ldin<BF16>(vsrc, ((k.tok0 + j) * p.G + g) * N + n) : 0.f;
      if (BF16)
        Vh[j * kBP + n] = __float2bfloat16_rn(v);  // exact
      else
        split_rn(v, Vh[j * kBP + n], Vl[j * kBP + n]);
    }
  }

  const int r16 = 16 * (w & 3), c64 = 64 * (w >> 2);
  const int gq = lane >> 2, tq = lane & 3;
  const LaneOff lo = lane_off(lane);
  for (int hh = 0; hh < nh; ++hh) {
    const int h = hb + hh;
    if (w == 0) weights(h);
    if (p.vec) tc::cp_async_wait_all();
    __syncthreads();  // weights, staged rows (and V) visible; the previous head's product is done
    if (p.vec) {
#pragma unroll
      for (int r = 0; r < kQb * kPmax / 4 / kThr; ++r) {
        const int e4 = t + kThr * r, j = e4 >> 4, q = (e4 & 15) * 4;
        const float m = sc[j];
        float4 v;
        if (kUB) {
          const uint2 b = *reinterpret_cast<const uint2*>(stg + 2 * (j * kPmax + q));
          v.x = __uint_as_float(b.x << 16);
          v.y = __uint_as_float(b.x & 0xffff0000u);
          v.z = __uint_as_float(b.y << 16);
          v.w = __uint_as_float(b.y & 0xffff0000u);
        } else {
          v = *reinterpret_cast<const float4*>(stg + 4 * (j * kPmax + q));
        }
        v.x *= m;
        v.y *= m;
        v.z *= m;
        v.w *= m;
        store_split4(Uh + j * kAP + q, Ul + j * kAP + q, v);
      }
    } else {
      for (int e = t; e < kQb * kPmax; e += kThr) {
        const int j = e / kPmax, q = e % kPmax;
        float v = 0.f;
        if (j < len && q < P) {
          const long long i = ((k.tok0 + j) * p.H + h) * P + q;
          v = sc[j] * (MODE == 0 ? ldin<BF16>(p.x, i) : p.dy[i]);
        }
        split_rn(v, Uh[j * kAP + q], Ul[j * kAP + q]);
      }
    }
    if (w == 0 && hh + 1 < nh) load_dt(h + 1);
    __syncthreads();  // U ready; the staging buffer is free
    if (p.vec && hh + 1 < nh) stage_u(h + 1);
    float* out = (MODE == 0 ? p.st : p.ad) + ((long long)c * p.H + h) * (long long)(P * N);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {  // 32 columns at a time
      const int cb = c64 + 32 * half;
      float acc[4][4];
      zero_acc(acc);
      if (r16 < P && cb < N)
        warp_mma<4, kAP, true, true, kBP, true, !BF16>(acc, acc, tc::smem_u32(Uh), tc::smem_u32(Ul),
                                                       r16, tc::smem_u32(Vh), tc::smem_u32(Vl), cb,
                                                       0, (len + 15) & ~15, lo);
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int n = cb + 8 * tt + 2 * tq;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int q = r16 + gq + 8 * hf;
          if (q < P) {
            if (p.vec) {
              if (n < N) *reinterpret_cast<float2*>(out + q * N + n) = make_float2(acc[tt][2 * hf], acc[tt][2 * hf + 1]);
            } else {
              if (n < N) out[q * N + n] = acc[tt][2 * hf];
              if (n + 1 < N) out[q * N + n + 1] = acc[tt][2 * hf + 1];
            }
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- passes
// FORWARD: st[c] <- state entering chunk c (from init); the state after the
// row's last chunk is not needed.  BACKWARD: ad[c] <- adjoint leaving chunk c
// (from dL/dfinal after the last chunk); dinit <- adjoint entering chunk 0.
template <bool FORWARD>
__global__ void __launch_bounds__(kThr) bwd_pass_kernel(BP p) {
  // one thread per float4 of a state; the chunks' values are independent
  // loads, issued eight at a time ahead of the recurrence
  const int PN = p.P * p.N;
  const int e4 = blockIdx.x * kThr + threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  if (4 * e4 >= PN) return;
  const long long sh = ((long long)b * p.H + h) * PN + 4 * e4;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (FORWARD && p.init) v = *reinterpret_cast<const float4*>(p.init + sh);
  if (!FORWARD && p.dfinal) v = *reinterpret_cast<const float4*>(p.dfinal + sh);
  float* buf = FORWARD ? p.st : p.ad;
  for (int i0 = 0; i0 < p.nc; i0 += 8) {
    float4 s[8];
    float d[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (i0 + u < p.nc) {
        const int c = b * p.nc + (FORWARD ? i0 + u : p.nc - 1 - (i0 + u));
        s[u] = __ldcg(reinterpret_cast<const float4*>(buf + ((long long)c * p.H + h) * PN + 4 * e4));
        d[u] = p.dec[(long long)c * p.H + h];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (i0 + u < p.nc) {
        const int c = b * p.nc + (FORWARD ? i0 + u : p.nc - 1 - (i0 + u));
        __stcg(reinterpret_cast<float4*>(buf + ((long long)c * p.H + h) * PN + 4 * e4), v);
        v.x = fmaf(d[u], v.x, s[u].x);
        v.y = fmaf(d[u], v.y, s[u].y);
        v.z = fmaf(d[u], v.z, s[u].z);
        v.w = fmaf(d[u], v.w, s[u].w);
      }
    }
  }
  if (!FORWARD && p.dinit) *reinterpret_cast<float4*>(p.dinit + sh) = v;
}

// ---------------------------------------------------------------- gradients
constexpr int kPP = kPmax + 1;  // padded row pitches
constexpr int kNP = kNmax + 1;
constexpr int kQP = kQb + 1;
constexpr int kTP = kNT + 1;
constexpr size_t kGradSmem = sizeof(float) * (2 * kQb * kPP + 2 * kQb * kNP + 3 * kQb * kQP +
                                              2 * kPmax * kTP + 8 * kQb);

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One block per (chunk, group, slice of kHS heads of the group): C B^T once,
// then head after head the gradients above; dB and dC of the slice's heads
// stay in registers and are added to global memory once.
template <bool BF16>
__global__ void __launch_bounds__(kThr) bwd_grad_kernel(BP p) {
  extern __shared__ float sm[];
  float* xs = sm;                  // [64][P+1] x rows
  float* dys = xs + kQb * kPP;     // [64][P+1] dy rows
  float* bs = dys + kQb * kPP;     // [64][N+1] B rows
  float* cs = bs + kQb * kNP;      // [64][N+1] C rows
  float* gs = cs + kQb * kNP;      // [64][65] G = C B^T
  float* mm = gs + kQb * kQP;      // [64][65] M
  float* gg = mm + kQb * kQP;      // [64][65] dG
  float* hs = gg + kQb * kQP;      // [P][33] tile of H_c
  float* dhs = hs + kPmax * kTP;   // [P][33] tile of dH_{c+1}
  float* cum = dhs + kPmax * kTP;  // [64]
  float* dts = cum + kQb;          // [64] dt
  float* ec = dts + kQb;           // [64] exp(cum_i)
  float* wt = ec + kQb;            // [64] w_j
  float* dcum = wt + kQb;          // [64] dL/dcum
  float* ddd = dcum + kQb;         // [64] direct dt terms
  float* red = ddd + kQb;          // [64] block reductions
  __shared__ float wsum[2];
  const int c = blockIdx.x, g = blockIdx.y;
  const Chunk k = chunk_of(p, c);
  const int P = p.P, N = p.N, len = k.len;
  const int hpg = p.H / p.G;
  const int hb = g * hpg + blockIdx.z * kHS;
  const int nh = min(kHS, hpg - blockIdx.z * kHS);
  const int t = threadIdx.x;
  const int ti = t >> 4, tj = t & 15;

  for (int e = t; e < kQb * N; e += kThr) {
    const int j = e / N, n = e % N;
    const bool ok = j < len;
    const long long i = ((k.tok0 + j) * p.G + g) * N + n;
    bs[j * kNP + n] = ok ? ldin<BF16>(p.B, i) : 0.f;
    cs[j * kNP + n] = ok ? ldin<BF16>(p.C, i) : 0.f;
  }
  __syncthreads();
  // G = C B^T; rows i = ti + 16 r, columns j = tj + 16 s
  {
    float gacc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) gacc[r][s2] = 0.f;
    for (int n = 0; n < N; ++n) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = cs[(ti + 16 * r) * kNP + n];
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) b[s2] = bs[(tj + 16 * s2) * kNP + n];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) gacc[r][s2] = fmaf(a[r], b[s2], gacc[r][s2]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) gs[(ti + 16 * r) * kQP + tj + 16 * s2] = gacc[r][s2];
  }
  // dB (rows j = ti + 16 r) and dC (rows i = ti + 16 r), columns n = tj + 16 s,
  // summed over the slice's heads
  float dca[4][8], dba[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) dca[r][s2] = dba[r][s2] = 0.f;

  for (int hh = 0; hh < nh; ++hh) {
    const int h = hb + hh;
    const float Ah = p.A[h];
    const float Dh = p.D ? p.D[h] : 0.f;
    __syncthreads();  // the previous head's tiles and tables are no longer read
    chunk_cum<BF16>(p, k, h, Ah, cum, dts, wsum);
    const float last = cum[len - 1];
    if (t < kQb) {
      ec[t] = expf(cum[t]);
      wt[t] = expf(last - cum[t]) * dts[t];
      dcum[t] = 0.f;
      ddd[t] = 0.f;
    }
    for (int e = t; e < kQb * P; e += kThr) {
      const int j = e / P, q = e % P;
      const bool ok = j < len;
      const long long i = ((k.tok0 + j) * p.H + h) * P + q;
      xs[j * kPP + q] = ok ? ldin<BF16>(p.x, i) : 0.f;
      dys[j * kPP + q] = ok ? p.dy[i] : 0.f;
    }
    __syncthreads();

    // ---- dS = dY X^T; M, dG and the decay terms of the quadratic form
    {
      float sacc[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) sacc[r][s2] = 0.f;
      for (int q = 0; q < P; ++q) {
        float a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = dys[(ti + 16 * r) * kPP + q];
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) b[s2] = xs[(tj + 16 * s2) * kPP + q];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2) sacc[r][s2] = fmaf(a[r], b[s2], sacc[r][s2]);
      }
      float rowT[4] = {0.f, 0.f, 0.f, 0.f}, colT[4] = {0.f, 0.f, 0.f, 0.f},
            colU[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = ti + 16 * r;
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
          const int j = tj + 16 * s2;
          float Mv = 0.f, dGv = 0.f;
          if (j <= i && i < len) {
            const float L = expf(cum[i] - cum[j]);
            const float GL = gs[i * kQP + j] * L;
            Mv = GL * dts[j];
            dGv = sacc[r][s2] * L * dts[j];
            const float T = sacc[r][s2] * Mv;
            rowT[r] += T;
            colT[s2] += T;
            colU[s2] += sacc[r][s2] * GL;
          }
          mm[i * kQP + j] = Mv;
          gg[i * kQP + j] = dGv;
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float v = half_warp_sum(rowT[r]);
        if (tj == 0) atomicAdd(&dcum[ti + 16 * r], v);
      }
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) {
        atomicAdd(&dcum[tj + 16 * s2], -colT[s2]);
        atomicAdd(&ddd[tj + 16 * s2], colU[s2]);
      }
    }
    __syncthreads();

    // ---- dX (intra) = M^T dY; rows j = ti + 16 r, columns q = tj + 16 s
    float dxa[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) dxa[r][s2] = 0.f;
    for (int i = 0; i < len; ++i) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = mm[i * kQP + ti + 16 * r];
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) b[s2] = tj + 16 * s2 < P ? dys[i * kPP + tj + 16 * s2] : 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) dxa[r][s2] = fmaf(a[r], b[s2], dxa[r][s2]);
    }
    // ---- dC += dG B, dB += dG^T C
    for (int jj = 0; jj < len; ++jj) {
      float a[4], a2[4], b[8], c2[8];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = gg[(ti + 16 * r) * kQP + jj];
        a2[r] = gg[jj * kQP + ti + 16 * r];
      }
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        b[s2] = bs[jj * kNP + tj + 16 * s2];
        c2[s2] = cs[jj * kNP + tj + 16 * s2];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          dca[r][s2] = fmaf(a[r], b[s2], dca[r][s2]);
          dba[r][s2] = fmaf(a2[r], c2[s2], dba[r][s2]);
        }
    }

    // ---- state terms, over tiles of 32 dstate columns:
    //   V = B dH^T (rows j, columns q), W = X dH, Z = dY H (rows, columns n), <dH, H>
    const float* Hc = p.st + ((long long)c * p.H + h) * (long long)(P * N);
    const float* dHc = p.ad + ((long long)c * p.H + h) * (long long)(P * N);
    float va[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) va[r][s2] = 0.f;
    float hdot = 0.f, zc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < kNmax / kNT; ++m) {
      const int n0 = m * kNT;
      if (n0 >= N) break;
      const int nt = min(kNT, N - n0);
      __syncthreads();
      for (int e = t; e < P * kNT; e += kThr) {
        const int q = e / kNT, nn = e % kNT;
        const bool ok = nn < nt;
        const float hv = ok ? __ldcg(Hc + (long long)q * N + n0 + nn) : 0.f;
        const float dv = ok ? __ldcg(dHc + (long long)q * N + n0 + nn) : 0.f;
        hs[q * kTP + nn] = hv;
        dhs[q * kTP + nn] = dv;
        hdot = fmaf(hv, dv, hdot);
      }
      __syncthreads();
      for (int nn = 0; nn < nt; ++nn) {
        float a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = bs[(ti + 16 * r) * kNP + n0 + nn];
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) b[s2] = tj + 16 * s2 < P ? dhs[(tj + 16 * s2) * kTP + nn] : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2) va[r][s2] = fmaf(a[r], b[s2], va[r][s2]);
      }
      float wa[4][2], za[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) wa[r][0] = wa[r][1] = za[r][0] = za[r][1] = 0.f;
      for (int q = 0; q < P; ++q) {
        float xa[4], ya[4], dh[2], hh2[2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          xa[r] = xs[(ti + 16 * r) * kPP + q];
          ya[r] = dys[(ti + 16 * r) * kPP + q];
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          dh[u] = dhs[q * kTP + tj + 16 * u];
          hh2[u] = hs[q * kTP + tj + 16 * u];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            wa[r][u] = fmaf(xa[r], dh[u], wa[r][u]);
            za[r][u] = fmaf(ya[r], hh2[u], za[r][u]);
          }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = ti + 16 * r;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int s2 = 2 * m + u;
          if (s2 < 8 && n0 + tj + 16 * u < N) {
            dba[r][s2] = fmaf(wt[row], wa[r][u], dba[r][s2]);
            const float zz = ec[row] * za[r][u];
            dca[r][s2] += zz;
            zc[r] = fmaf(zz, cs[row * kNP + n0 + tj + 16 * u], zc[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float v = half_warp_sum(zc[r]);
      if (tj == 0) atomicAdd(&dcum[ti + 16 * r], v);
    }
    float wv_sum = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = ti + 16 * r;
      float vj = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2)
        if (tj + 16 * s2 < P) vj = fmaf(xs[j * kPP + tj + 16 * s2], va[r][s2], vj);
      vj = half_warp_sum(vj);
      if (tj == 0 && j < len) {
        atomicAdd(&dcum[j], -wt[j] * vj);
        atomicAdd(&ddd[j], expf(last - cum[j]) * vj);
        wv_sum = fmaf(wt[j], vj, wv_sum);
      }
    }
    // dx = M^T dy + w_j dH B_j + D dy
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = ti + 16 * r;
      if (j < len) {
        float* dst = p.dx + ((k.tok0 + j) * p.H + h) * P;
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
          const int q = tj + 16 * s2;
          if (q < P) dst[q] = dxa[r][s2] + wt[j] * va[r][s2] + Dh * dys[j * kPP + q];
        }
      }
    }
    // block sums: <dH, H>, sum_j w_j v_j, dD
    float dd = 0.f;
    for (int e = t; e < len * P; e += kThr)
      dd = fmaf(dys[(e / P) * kPP + e % P], xs[(e / P) * kPP + e % P], dd);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      hdot += __shfl_xor_sync(0xffffffffu, hdot, o);
      wv_sum += __shfl_xor_sync(0xffffffffu, wv_sum, o);
      dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    if ((t & 31) == 0) {
      red[t >> 5] = hdot;
      red[8 + (t >> 5)] = wv_sum;
      red[16 + (t >> 5)] = dd;
    }
    __syncthreads();
    if (t == 0) {
      float a = 0.f, b = 0.f, d2 = 0.f;
      for (int w = 0; w < kThr / 32; ++w) {
        a += red[w];
        b += red[8 + w];
        d2 += red[16 + w];
      }
      dcum[len - 1] += expf(last) * a + b;
      if (p.dD) atomicAdd(p.dD + h, d2);
    }
    __syncthreads();
    // ddt_j = direct terms + A sum_{k>=j} dcum_k; dA += sum_j dt_j sum_{k>=j} dcum_k
    if (t < 32) {
      // reverse inclusive scan over the 64 entries, two per lane (lane l owns
      // entries 63 - 2l and 62 - 2l, the later one first)
      const int j1 = kQb - 1 - 2 * t, j2 = j1 - 1;
      const float a1 = dcum[j1], a2 = dcum[j2];
      float v = a1 + a2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (t >= o) v += u;
      }
      const float r2 = v;       // sum over k >= j2
      const float r1 = v - a2;  // sum over k >= j1
      float da = 0.f;
      if (j1 < len) {
        p.ddt[(k.tok0 + j1) * p.H + h] = ddd[j1] + Ah * r1;
        da = fmaf(dts[j1], r1, da);
      }
      if (j2 < len) {
        p.ddt[(k.tok0 + j2) * p.H + h] = ddd[j2] + Ah * r2;
        da = fmaf(dts[j2], r2, da);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
      if (t == 0) atomicAdd(p.dA + h, da);
    }
  }
  // dB, dC of the slice's heads
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = ti + 16 * r;
    if (j < len) {
      float* db = p.dB + ((k.tok0 + j) * p.G + g) * N;
      float* dc = p.dC + ((k.tok0 + j) * p.G + g) * N;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        const int n = tj + 16 * s2;
        if (n < N) {
          atomicAdd(db + n, dba[r][s2]);
          atomicAdd(dc + n, dca[r][s2]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- gradients, tcgen05
// The gradient kernel on the fifth-generation tensor cores (bf16 inputs,
// headdim and dstate multiples of 8).  Per block (chunk, group, slice of up
// to kHS heads of the group), 16 math warps and one MMA warp.  Operands are
// 128-byte-swizzled bf16 tiles of 64 rows (exact for x, B, C; hi/lo pairs
// for dy, exp(cum) dy, w x, H_c, dH_{c+1}, M and dG; H_c and dH_{c+1} come
// split and transposed, 128 rows of dstate, from the state scans by TMA
// loads a head ahead), zero-padded to headdim 64 and dstate 128, read by the
// MMAs K-major or MN-major as each product needs.  Accumulators, summed
// over the slice's heads, transposed (M = 128: dstate row n in TMEM lane n;
// 128 columns, token j in columns j and 64 + j, the products with the two
// halves of a stacked hi/lo operand):
//   dC^T += H^T (exp(cum) dY)^T + B^T dG^T          dB^T += dH^T (w o X)^T + C^T dG
// and per head (M = 64: row r in TMEM lane 32 (r / 16) + r % 16):
//   S  = dY X^T (the first head's C B^T before it)   V = B dH^T
//   Xi = M^T dY (D on M's diagonal: + D dy)          U = C H^T
// Per head: operands -> smem; MMAs dS, V, U, dC, dB; the dS epilogue writes M
// and dG; MMAs Xi, dC, dB; the epilogue of V, U, Xi writes dx and the decay
// terms, and the next head's H, dH loads start; warp 0 closes ddt and dA.  Every wait is bounded: one that runs out
// records SSD_ERR_TIMEOUT and the block goes on (its results are then
// undefined) and waits once more for its last MMAs before freeing TMEM.
namespace tg {
constexpr int kMathWarps = 16;
constexpr int kThreads = 32 * (kMathWarps + 1);
constexpr int kMathThreads = 32 * kMathWarps;
constexpr uint32_t kAtom = 8192;  // 64 rows x 128 bytes
constexpr uint32_t oB = 0, oC = 2 * kAtom, oX = 4 * kAtom, oWXh = 5 * kAtom, oWXl = 6 * kAtom,
                   oYh = 7 * kAtom, oYl = 8 * kAtom, oEYh = 9 * kAtom, oEYl = 10 * kAtom,
                   oHh = 11 * kAtom, oHl = 13 * kAtom, oDh = 15 * kAtom, oDl = 17 * kAtom,
                   oMh = 19 * kAtom, oMl = 20 * kAtom, oGh = 21 * kAtom, oGl = 22 * kAtom,
                   oTab = 23 * kAtom;
// tables (floats): two buffers of (log2e cum, exp(cum), w, exp(cum_last -
// cum)) [64]; per head of the slice dt [kHS][64]; per head the partial decay
// sums, each slot with one writer: dL/dcum by row and column group [4][64],
// the direct dt terms by row and column group [4][64] and by column and row
// group [4][64]; log2e cum_last [kHS][4] (every fourth); log2e A [kHS]; and
// per warp (one writer each) the partial sums of <dH, H>, sum_j w_j v_j and
// dD [kHS][3][16]
constexpr uint32_t kPart = 3 * 4 * kQb;  // partial sums per head
constexpr uint32_t kTabFloats = 2 * 4 * kQb + kHS * kQb + kHS * kPart + 4 * kHS + kHS + 48 * kHS;
constexpr uint32_t oBar = oTab + 4 * kTabFloats;
constexpr uint32_t kSmem = oBar + 64 + 1024;  // + alignment of the tiles to 1024 bytes
static_assert(kSmem <= 232448, "shared memory per block");
constexpr uint32_t cDC = 0, cDB = 128, cS = 256, cX = 320, cV = 384, cU = 448;  // TMEM columns
constexpr uint32_t kIdKK64 = tc::idesc_bf16(64, 64, false, false);
constexpr uint32_t kIdNN64 = tc::idesc_bf16(64, 64, true, true);
// the transposed dC, dB products: M = 128 (dstate), N = 128 (a stacked hi/lo
// operand) or 64
constexpr uint32_t kIdT128 = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdT64 = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdTMK = tc::idesc_bf16(128, 128, true, false);
constexpr uint32_t kIdTMM = tc::idesc_bf16(128, 128, true, true);
constexpr uint32_t kIdKN64 = tc::idesc_bf16(64, 64, false, true);
constexpr float kLog2e = 1.4426950408889634f;

// byte offset of element (r, c) of a 64-row tile made of 64-column atoms
__device__ __forceinline__ uint32_t swo(int r, int c) {
  return (uint32_t)(c >> 6) * kAtom + tc::sw128_offset(r, (c & 63) >> 3) + (c & 7) * 2;
}
// descriptor offsets (16-byte units) of k-step kk: K-major +32 bytes inside
// an atom, atoms kAtom apart; MN-major +16 rows (64-element MN blocks kAtom
// apart, the descriptor's leading offset)
__host__ __device__ constexpr uint64_t kof(int kk) { return (uint64_t)((kk >> 2) * (kAtom >> 4) + (kk & 3) * 2); }
__host__ __device__ constexpr uint64_t mof(int kk) { return (uint64_t)(kk * 128); }
// 16 lanes x 16 columns: per thread the m16n8 accumulator fragments of the
// warp's 16 rows (rows lane/4 and lane/4 + 8, columns 8 b + 2 (lane % 4) +
// {0, 1} of block b = 0, 1)
__device__ __forceinline__ void ld_frag2(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// a pair of fp32 -> bf16 hi = rn(v), lo = rn(v - hi), packed (x in the low half)
__device__ __forceinline__ void split2rn(tc::f2 v, uint32_t& hi, uint32_t& lo) {
  hi = tc::pack_bf16(v.x, v.y);
  const tc::f2 r = tc::sub2(v, tc::bf2(hi));
  lo = tc::pack_bf16(r.x, r.y);
}
// eight fp32 (four pairs) -> hi/lo, 16 bytes each
__device__ __forceinline__ void split8(const tc::f2 (&v)[4], uint4& hi, uint4& lo) {
  split2rn(v[0], hi.x, lo.x);
  split2rn(v[1], hi.y, lo.y);
  split2rn(v[2], hi.z, lo.z);
  split2rn(v[3], hi.w, lo.w);
}
// four fp32 -> hi/lo, 8 bytes each, at byte addresses ph / pl
__device__ __forceinline__ void split4_at(unsigned char* ph, unsigned char* pl, float4 v) {
  uint2 hi, lo;
  split2rn(tc::f2{v.x, v.y}, hi.x, lo.x);
  split2rn(tc::f2{v.z, v.w}, hi.y, lo.y);
  *reinterpret_cast<uint2*>(ph) = hi;
  *reinterpret_cast<uint2*>(pl) = lo;
}
__device__ __forceinline__ tc::f2 bf2_at(const unsigned char* p) {
  return tc::bf2(*reinterpret_cast<const uint32_t*>(p));
}
}  // namespace tg

// A bounded mbarrier wait that gives up at once when an earlier wait of the
// block ran out (*abort), and raises *abort when it runs out itself: a
// block whose wait expired unwinds without waiting again.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                      uint32_t polls) {
  if (*abort) return false;
  if (tc::mbar_wait(bar, parity, polls)) return true;
  *abort = 1;
  return false;
}

__global__ void __launch_bounds__(tg::kThreads, 1)
    bwd_grad_tc_kernel(BP p, const __grid_constant__ CUtensorMap map_hh,
                       const __grid_constant__ CUtensorMap map_hl,
                       const __grid_constant__ CUtensorMap map_dh,
                       const __grid_constant__ CUtensorMap map_dl) {
  using namespace tg;
  using tc::f2;
  extern __shared__ unsigned char tsm_raw[];
  const uint32_t raw_s = tc::smem_u32(tsm_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  unsigned char* base = tsm_raw + (sb - raw_s);
  float* tabs = reinterpret_cast<float*>(base + oTab);
  float* dtsH = tabs + 8 * kQb;          // [kHS][64] dt per head (after the two 4 x 64 table buffers)
  float* partH = dtsH + kHS * kQb;       // [kHS][kPart] partial decay sums per head
  float* hsum = partH + kHS * kPart;     // [kHS][4] per head
  float* atab = hsum + 4 * kHS;          // [kHS] log2e A per head
  float* wsum = atab + kHS;              // [kHS][3][16] per-warp sums: <dH, H>, sum w v, dD
  // mbarriers, one phase per head each: C B^T (once), dS, group 1, group 2,
  // Xi; then the drain of the last MMAs (once); and the TMA loads of H, dH
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + oBar);
  uint32_t* tptr = reinterpret_cast<uint32_t*>(base + oBar + 48);
  volatile int* abort_f = reinterpret_cast<volatile int*>(base + oBar + 52);
  uint64_t* hdbar = reinterpret_cast<uint64_t*>(base + oBar + 56);
  const int c = blockIdx.x, g = blockIdx.y;
  const Chunk k = chunk_of(p, c);
  const int P = p.P, N = p.N, len = k.len;
  const int hpg = p.H / p.G;
  const int hb = g * hpg + blockIdx.z * kHS;
  const int nh = min(kHS, hpg - blockIdx.z * kHS);
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const bool math = w < kMathWarps;
  const int gq = lane >> 2, tq = lane & 3;
  const int qd = w & 3, cg = w >> 2;  // math warps: TMEM lane quadrant (rows 16 qd..), column group
  const int r16 = 16 * qd, c16 = 16 * cg;
  const uint32_t lanebase = (uint32_t)(32 * qd) << 16;
  const __nv_bfloat16* xg = reinterpret_cast<const __nv_bfloat16*>(p.x);
  bool ok = true;  // every wait of this thread completed

  // One head's x and dy in registers (zero outside the valid rows and
  // headdim), loaded a head ahead of their use.  Math thread t: row t / 8,
  // columns 8 (t % 8)..
  uint4 vx = make_uint4(0, 0, 0, 0);
  float4 vy[2];
  const auto load_head = [&](int h) {
    const int j = t >> 3, q = (t & 7) * 8;
    const bool okr = j < len && q < P;
    const long long row = ((k.tok0 + j) * p.H + h) * P + q;
    vx = okr ? *reinterpret_cast<const uint4*>(xg + row) : make_uint4(0, 0, 0, 0);
    vy[0] = okr ? *reinterpret_cast<const float4*>(p.dy + row) : make_float4(0.f, 0.f, 0.f, 0.f);
    vy[1] = okr ? *reinterpret_cast<const float4*>(p.dy + row + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // H_c and dH_{c+1} of slice head hh (bf16 hi/lo pairs of the transposed
  // states, as the state scans stored them) into their operand tiles by TMA,
  // zero past dstate and headdim; completes phase hh of hdbar.  One thread.
  const auto load_hd = [&](int hh) {
    const int slab = (int)((long long)c * p.H + hb + hh);
    tc::mbar_arrive_expect_tx(hdbar, 8u * kAtom);
    tc::tma_load_3d(base + oHh, &map_hh, hdbar, 0, 0, slab);
    tc::tma_load_3d(base + oHh + kAtom, &map_hh, hdbar, 0, 64, slab);
    tc::tma_load_3d(base + oHl, &map_hl, hdbar, 0, 0, slab);
    tc::tma_load_3d(base + oHl + kAtom, &map_hl, hdbar, 0, 64, slab);
    tc::tma_load_3d(base + oDh, &map_dh, hdbar, 0, 0, slab);
    tc::tma_load_3d(base + oDh + kAtom, &map_dh, hdbar, 0, 64, slab);
    tc::tma_load_3d(base + oDl, &map_dl, hdbar, 0, 0, slab);
    tc::tma_load_3d(base + oDl + kAtom, &map_dl, hdbar, 0, 64, slab);
  };
  int hd_issued = 0;  // MMA warp, lane 0: heads whose H, dH loads it issued
  const auto prefetch_head = [&](int h) {
    const long long sOff = ((long long)c * p.H + h) * (long long)(P * N);
    if (t == 0) {
      tc::bulk_prefetch_l2(p.sth + sOff, (uint32_t)(P * N * 2));
      tc::bulk_prefetch_l2(p.stl + sOff, (uint32_t)(P * N * 2));
      tc::bulk_prefetch_l2(p.adh + sOff, (uint32_t)(P * N * 2));
      tc::bulk_prefetch_l2(p.adl + sOff, (uint32_t)(P * N * 2));
    } else if (t >= 32 && t < 32 + kQb && t - 32 < len) {
      const long long row = (k.tok0 + (t - 32)) * p.H + h;
      tc::prefetch_l2(xg + row * P);
      tc::prefetch_l2(p.dy + row * P);
      if (P > 32) tc::prefetch_l2(p.dy + row * P + 32);
    }
  };
  // One warp: the decay tables of slice head hh into buffer hh % 2 (lane l:
  // rows 2l, 2l+1) and its log2e cum_last, from the head's dt and A staged in
  // shared memory by the prologue (head 0: from global memory, `fromg`).
  const auto tables = [&](int hh, bool fromg) {
    const int h = hb + hh;
    float* c2 = tabs + 4 * (hh & 1) * kQb;
    float* ec = c2 + kQb;
    float* wt = ec + kQb;
    float* el = wt + kQb;
    const float Ah = fromg ? p.A[h] * kLog2e : atab[hh];
    const int j0 = 2 * lane, j1 = j0 + 1;
    const float d0 = fromg ? (j0 < len ? ldin<true>(p.dt, (k.tok0 + j0) * p.H + h) : 0.f)
                           : dtsH[hh * kQb + j0];
    const float d1 = fromg ? (j1 < len ? ldin<true>(p.dt, (k.tok0 + j1) * p.H + h) : 0.f)
                           : dtsH[hh * kQb + j1];
    const float a1 = d1 * Ah;
    float s = d0 * Ah + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    const float cm1 = s, cm0 = s - a1;
    const float lst = __shfl_sync(0xffffffffu, ((len - 1) & 1) ? cm1 : cm0, (len - 1) >> 1);
    c2[j0] = cm0;
    c2[j1] = cm1;
    dtsH[hh * kQb + j0] = d0;
    dtsH[hh * kQb + j1] = d1;
    ec[j0] = tc::fast_exp2(cm0);
    ec[j1] = tc::fast_exp2(cm1);
    const float e0 = tc::fast_exp2(lst - cm0), e1 = tc::fast_exp2(lst - cm1);
    el[j0] = e0;
    el[j1] = e1;
    wt[j0] = e0 * d0;
    wt[j1] = e1 * d1;
    if (lane == 0) hsum[4 * hh] = lst;
  };

  // The operands of slice head hh read only by the first MMA group besides
  // H and dH: w o x and exp(cum) o dy (hi/lo) from the registers (x, dy of
  // that head) and its tables; the block sum dD of the head.  Math threads.
  const auto store_early = [&](int hh) {
    const float* ec = tabs + (4 * (hh & 1) + 1) * kQb;
    const float* wt = ec + kQb;
    const int j = t >> 3, q = (t & 7) * 8;
    const uint32_t o8 = swo(j, q);
    const f2 xf[4] = {tc::bf2(vx.x), tc::bf2(vx.y), tc::bf2(vx.z), tc::bf2(vx.w)};
    const f2 yf[4] = {f2{vy[0].x, vy[0].y}, f2{vy[0].z, vy[0].w}, f2{vy[1].x, vy[1].y},
                      f2{vy[1].z, vy[1].w}};
    const f2 wj{wt[j], wt[j]}, ej{ec[j], ec[j]};
    f2 sx[4], sy[4], dd2{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dd2 = tc::fma2(xf[i], yf[i], dd2);
      sx[i] = tc::mul2(wj, xf[i]);
      sy[i] = tc::mul2(ej, yf[i]);
    }
    uint4 hi, lo;
    split8(sx, hi, lo);
    *reinterpret_cast<uint4*>(base + oWXh + o8) = hi;
    *reinterpret_cast<uint4*>(base + oWXl + o8) = lo;
    split8(sy, hi, lo);
    *reinterpret_cast<uint4*>(base + oEYh + o8) = hi;
    *reinterpret_cast<uint4*>(base + oEYl + o8) = lo;
    tc::fence_proxy_async_smem();
    float dd = dd2.x + dd2.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
    if (lane == 0) wsum[(hh * 3 + 2) * 16 + w] = dd;
  };
  // <dH_{c+1}, H_c> of slice head hh from its operand tiles (hi + lo; both
  // tiles share one layout, so equal offsets hold matching elements), by
  // five warps (index iw), after the tiles' TMA loads completed.
  const auto hdot_tiles = [&](int hh, int iw) {
    float hd = 0.f;
#pragma unroll 1
    for (int k16 = 32 * iw + lane; k16 < (int)(2 * kAtom / 16); k16 += 5 * 32) {
      const uint32_t o = 16u * (uint32_t)k16;
      const uint4 a = *reinterpret_cast<const uint4*>(base + oHh + o);
      const uint4 b = *reinterpret_cast<const uint4*>(base + oHl + o);
      const uint4 d = *reinterpret_cast<const uint4*>(base + oDh + o);
      const uint4 e = *reinterpret_cast<const uint4*>(base + oDl + o);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      const uint32_t dw[4] = {d.x, d.y, d.z, d.w}, ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 hv = tc::add2(tc::bf2(aw[i]), tc::bf2(bw[i]));
        const f2 dv = tc::add2(tc::bf2(dw[i]), tc::bf2(ew[i]));
        hd = fmaf(hv.x, dv.x, fmaf(hv.y, dv.y, hd));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, o);
    if (lane == 0) wsum[hh * 3 * 16 + iw] = hd;
  };

  // ---- prologue: B, C tiles; the first head's operands and tables; TMEM; C B^T
  if (math) {
    const __nv_bfloat16* Bg = reinterpret_cast<const __nv_bfloat16*>(p.B);
    const __nv_bfloat16* Cg = reinterpret_cast<const __nv_bfloat16*>(p.C);
    uint4 vb[2], vc[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int e8 = t + kMathThreads * r, j = e8 >> 4, n = (e8 & 15) * 8;
      const bool okb = j < len && n < N;
      const long long i = ((k.tok0 + j) * p.G + g) * N + n;
      vb[r] = okb ? *reinterpret_cast<const uint4*>(Bg + i) : make_uint4(0, 0, 0, 0);
      vc[r] = okb ? *reinterpret_cast<const uint4*>(Cg + i) : make_uint4(0, 0, 0, 0);
    }
    load_head(hb);
    if (nh > 1) prefetch_head(hb + 1);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int e8 = t + kMathThreads * r, j = e8 >> 4, n = (e8 & 15) * 8;
      *reinterpret_cast<uint4*>(base + oB + swo(j, n)) = vb[r];
      *reinterpret_cast<uint4*>(base + oC + swo(j, n)) = vc[r];
    }
    for (int e = t; e < (int)(kHS * kPart + 4 * kHS); e += kMathThreads) partH[e] = 0.f;  // partial sums
    // M and dG: the blocks above the diagonal stay zero (no warp writes them)
    for (int e = t; e < (int)(4 * kAtom / 16); e += kMathThreads)
      *reinterpret_cast<uint4*>(base + oMh + 16 * e) = make_uint4(0, 0, 0, 0);
    if (w == 0) {
      tables(0, true);
    } else {  // the other heads' dt and A, for their tables later
      for (int e = t - 32; e < (nh - 1) * kQb; e += kMathThreads - 32) {
        const int hh = 1 + e / kQb, j = e % kQb;
        dtsH[hh * kQb + j] = j < len ? ldin<true>(p.dt, (k.tok0 + j) * p.H + hb + hh) : 0.f;
      }
      if (t - 32 < nh) atab[t - 32] = p.A[hb + t - 32] * kLog2e;
    }
    tc::fence_proxy_async_smem();
  } else {
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < 6; ++i) tc::mbar_init(&bars[i], 1);
      tc::mbar_init(hdbar, 1);
      *abort_f = 0;
      tc::fence_mbar_init();
    }
    __syncwarp();
    tc::tmem_alloc(tptr, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tptr;
  if (w == kMathWarps && lane == 0) {  // the first head's H, dH
    load_hd(0);
    hd_issued = 1;
  }
  // operand descriptors: one K-major and one MN-major base, the tiles at
  // constant offsets from it (start-address field, 16-byte units)
  const uint64_t kd0 = tc::sdesc_sw128(sb, 16, 1024), md0 = tc::sdesc_sw128(sb, kAtom, 1024);
#define KD(off, kk) (kd0 + ((off) >> 4) + kof(kk))
#define MD(off, kk) (md0 + ((off) >> 4) + mof(kk))
  if (!math) {
    if (tc::elect_one()) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) tc::mma_bf16(tm + cS, KD(oC, kk), KD(oB, kk), kIdKK64, kk > 0);
      tc::mma_commit(&bars[0]);
    }
    __syncwarp();
  }
  float gr[8];  // C B^T at this thread's dS fragment positions
  if (math) {
    store_early(0);
    ok &= bwait(&bars[0], 0, abort_f, p.wait_polls);
    tc::tc_fence_after();
    ld_frag2(tm + lanebase + cS + c16, gr);
    tc::tmem_ld_wait();
    tc::tie8(gr);
  }

  for (int hh = 0; hh < nh; ++hh) {
    const int h = hb + hh;
    const uint32_t par = hh & 1;
    const float* c2 = tabs + 4 * (hh & 1) * kQb;  // log2e cum
    const float* ec = c2 + kQb;
    const float* wt = ec + kQb;
    const float* el = wt + kQb;
    const float* dts = dtsH + hh * kQb;
    float* rrow = partH + hh * kPart + cg * kQb;              // dL/dcum, rows, this column group
    float* drow = partH + hh * kPart + (4 + cg) * kQb;        // direct dt terms, rows
    float* dcol = partH + hh * kPart + (8 + qd) * kQb;        // direct dt terms, columns, this row group
    // ---- x and dy of this head to shared memory (H, dH, w o x and
    //      exp(cum) o dy went in while the previous head's second MMA group ran)
    if (math) {
      const int j = t >> 3, q = (t & 7) * 8;
      const uint32_t o8 = swo(j, q);
      *reinterpret_cast<uint4*>(base + oX + o8) = vx;
      const f2 yf[4] = {f2{vy[0].x, vy[0].y}, f2{vy[0].z, vy[0].w}, f2{vy[1].x, vy[1].y},
                        f2{vy[1].z, vy[1].w}};
      uint4 hi, lo;
      split8(yf, hi, lo);
      *reinterpret_cast<uint4*>(base + oYh + o8) = hi;
      *reinterpret_cast<uint4*>(base + oYl + o8) = lo;
      tc::fence_proxy_async_smem();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- group 1: dS = dY X^T; V = B dH^T; U = C H^T; dC^T += H^T (ec o dY)^T;
    //      dB^T += dH^T (w o X)^T
    if (!math) {
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_bf16(tm + cS, KD(oYh, kk), KD(oX, kk), kIdKK64, kk > 0);
          tc::mma_bf16(tm + cS, KD(oYl, kk), KD(oX, kk), kIdKK64, true);
        }
        if (!(p.hold == 1 && hh == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0))
          tc::mma_commit(&bars[1]);  // (the test hook holds back the first one of block 0)
        ok &= bwait(hdbar, par, abort_f, p.wait_polls);  // this head's H, dH in their tiles
        // (H^T and dH^T are the tiles as stored, K-major over headdim; the hi
        // and lo tiles of exp(cum) dy and of w x are adjacent: one operand of
        // N = 128)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const bool acc = hh > 0 || kk > 0;
          tc::mma_bf16(tm + cDC, KD(oHh, kk), KD(oEYh, kk), kIdT128, acc);
          tc::mma_bf16(tm + cDC, KD(oHl, kk), KD(oEYh, kk), kIdT64, true);
          tc::mma_bf16(tm + cDB, KD(oDh, kk), KD(oWXh, kk), kIdT128, acc);
          tc::mma_bf16(tm + cDB, KD(oDl, kk), KD(oWXh, kk), kIdT64, true);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          tc::mma_bf16(tm + cV, KD(oB, kk), MD(oDh, kk), kIdKN64, kk > 0);
          tc::mma_bf16(tm + cV, KD(oB, kk), MD(oDl, kk), kIdKN64, true);
          tc::mma_bf16(tm + cU, KD(oC, kk), MD(oHh, kk), kIdKN64, kk > 0);
          tc::mma_bf16(tm + cU, KD(oC, kk), MD(oHl, kk), kIdKN64, true);
        }
        tc::mma_commit(&bars[2]);
      }
      __syncwarp();
    } else {
      // ---- dS epilogue: M = G L dt (+ D on the diagonal), dG = dS L dt;
      //      the decay terms of the quadratic form (rows r16.., columns
      //      c16..), by the warps whose block meets the causal mask; of the
      //      others, warp 4 makes the next head's tables and five sum <dH, H>
      if (cg <= qd) {
        ok &= bwait(&bars[1], par, abort_f, p.wait_polls);
        tc::tc_fence_after();
        float sa[8];
        ld_frag2(tm + lanebase + cS + c16, sa);
        tc::tmem_ld_wait();
        tc::tie8(sa);
        const float Dd = p.D ? p.D[h] : 0.f;
        float rowT[2] = {0.f, 0.f}, colU[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        const float c2i[2] = {c2[r16 + gq], c2[r16 + gq + 8]};
        float c2j[4], dtj[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int j = c16 + 8 * (f >> 1) + 2 * tq + (f & 1);
          c2j[f] = c2[j];
          dtj[f] = dts[j];
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int i = r16 + gq + 8 * hf;
            float mv[2], dv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = c16 + 8 * tt + 2 * tq + e;
              const int f = 4 * tt + 2 * hf + e;
              mv[e] = dv[e] = 0.f;
              if (j <= i && i < len) {
                const float L = tc::fast_exp2(c2i[hf] - c2j[2 * tt + e]);
                const float GL = gr[f] * L;
                mv[e] = GL * dtj[2 * tt + e];
                dv[e] = sa[f] * L * dtj[2 * tt + e];
                rowT[hf] = fmaf(sa[f], mv[e], rowT[hf]);
                colU[tt][e] = fmaf(sa[f], GL, colU[tt][e]);
                if (i == j) mv[e] += Dd;
              }
            }
            uint32_t mh, ml, gh, gl;
            split2rn(f2{mv[0], mv[1]}, mh, ml);
            split2rn(f2{dv[0], dv[1]}, gh, gl);
            const uint32_t o = swo(i, c16 + 8 * tt + 2 * tq);
            *reinterpret_cast<uint32_t*>(base + oMh + o) = mh;
            *reinterpret_cast<uint32_t*>(base + oMl + o) = ml;
            *reinterpret_cast<uint32_t*>(base + oGh + o) = gh;
            *reinterpret_cast<uint32_t*>(base + oGl + o) = gl;
          }
        }
        tc::fence_proxy_async_smem();
        // partial sums, one writer per slot: rows (quad sums) and columns
        // (column j: sum_i dS M = dt_j sum_i dS G L; sums over the warp's rows)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float v = rowT[hf];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (tq == 0) rrow[r16 + gq + 8 * hf] = v;
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float b = colU[tt][e];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
            if (gq == 0) dcol[c16 + 8 * tt + 2 * tq + e] = b;
          }
      } else if (w != 4) {
        ok &= bwait(hdbar, par, abort_f, p.wait_polls);
        hdot_tiles(hh, cg == 2 ? qd : 2 + qd);
      } else if (hh + 1 < nh) {
        tables(hh + 1, false);
      }
      // the next head's x, dy into registers (this head's are in shared memory)
      if (hh + 1 < nh) {
        load_head(h + 1);
        if (hh + 2 < nh) prefetch_head(h + 2);
      }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- group 2: Xi = M^T dY; dC^T += B^T dG^T; dB^T += C^T dG
    if (!math) {
      if (tc::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_bf16(tm + cX, MD(oMh, kk), MD(oYh, kk), kIdNN64, kk > 0);
          tc::mma_bf16(tm + cX, MD(oMl, kk), MD(oYh, kk), kIdNN64, true);
          tc::mma_bf16(tm + cX, MD(oMh, kk), MD(oYl, kk), kIdNN64, true);
        }
        tc::mma_commit(&bars[4]);
        // (B^T, C^T: the tiles read MN-major; dG hi and lo adjacent: one
        // operand of N = 128, K-major for dC, MN-major for dB)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_bf16(tm + cDC, MD(oB, kk), KD(oGh, kk), kIdTMK, true);
          tc::mma_bf16(tm + cDB, MD(oC, kk), MD(oGh, kk), kIdTMM, true);
        }
        tc::mma_commit(&bars[3]);
      }
      __syncwarp();
      // once group 1 completed (the <dH, H> sums were done before the second
      // barrier), the H, dH tiles are free: the next head's go in, after this
      // head's loads completed (the phases of hdbar never overlap, even after
      // an expired wait)
      if (lane == 0 && hh + 1 < nh && hd_issued == hh + 1 &&
          tc::mbar_wait(&bars[2], par, p.wait_polls) &&
          tc::mbar_wait(hdbar, (uint32_t)(hh & 1), p.wait_polls)) {
        load_hd(hh + 1);
        hd_issued = hh + 2;
      }
      __syncwarp();
    } else {
      // ---- V, U: the state terms of the decay; then dx = Xi + w_j V
      ok &= bwait(&bars[2], par, abort_f, p.wait_polls);
      tc::tc_fence_after();
      float va[8], ua[8];
      ld_frag2(tm + lanebase + cV + c16, va);
      ld_frag2(tm + lanebase + cU + c16, ua);
      tc::tmem_ld_wait();
      tc::tie8(va);
      tc::tie8(ua);
      float vp[2] = {0.f, 0.f}, zc[2] = {0.f, 0.f};
#pragma unroll
      for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = r16 + gq + 8 * hf;
          const uint32_t o = swo(r, c16 + 8 * tt + 2 * tq);
          const f2 xv = bf2_at(base + oX + o);
          const f2 yv = tc::add2(bf2_at(base + oYh + o), bf2_at(base + oYl + o));
          const int f = 4 * tt + 2 * hf;
          vp[hf] += xv.x * va[f] + xv.y * va[f + 1];
          zc[hf] += yv.x * ua[f] + yv.y * ua[f + 1];
        }
      float wv_sum = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v = vp[hf], z = zc[hf];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        const int r = r16 + gq + 8 * hf;
        if (tq == 0) {
          const bool okr = r < len;
          rrow[r] += okr ? ec[r] * z - wt[r] * v : 0.f;  // this thread wrote the row's dS part
          drow[r] = okr ? el[r] * v : 0.f;
          if (okr) wv_sum = fmaf(wt[r], v, wv_sum);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wv_sum += __shfl_xor_sync(0xffffffffu, wv_sum, o);
      if (lane == 0) wsum[(hh * 3 + 1) * 16 + w] = wv_sum;
      // the first group is done with H, dH, w o x and exp(cum) o dy: the next
      // head's go in now (its tables came with the second barrier)
      if (hh + 1 < nh) store_early(hh + 1);
      // Xi (committed before the products into dC and dB)
      ok &= bwait(&bars[4], par, abort_f, p.wait_polls);
      tc::tc_fence_after();
      float xa[8];
      ld_frag2(tm + lanebase + cX + c16, xa);
      tc::tmem_ld_wait();
      tc::tie8(xa);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = r16 + gq + 8 * hf;
        const float wj = wt[j];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int q = c16 + 8 * tt + 2 * tq;
          const int f = 4 * tt + 2 * hf;
          if (j < len && q < P)
            *reinterpret_cast<float2*>(p.dx + ((k.tok0 + j) * p.H + h) * P + q) =
                make_float2(fmaf(wj, va[f], xa[f]), fmaf(wj, va[f + 1], xa[f + 1]));
        }
      }
      // group 2 complete before its operands are overwritten
      ok &= bwait(&bars[3], par, abort_f, p.wait_polls);
    }
    tc::tc_fence_before();
    __syncthreads();
  }
  tc::tc_fence_after();
  // ---- per head of the slice (warp hh): ddt_j = direct terms + A
  //      sum_{k>=j} dcum_k, with the state terms <dH, H> and sum_j w_j v_j
  //      at the last valid row; dA += sum_j dt_j sum_{k>=j} dcum_k; dD
  if (math && w < nh) {
    const int hh = w, h = hb + w;
    const float* dts = dtsH + hh * kQb;
    const float* part = partH + hh * kPart;
    // dL/dcum_j and the direct dt terms from the partial sums
    const auto sums = [&](int j, float& dc, float& dd) {
      float r = 0.f, d = 0.f, cu = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        r += part[k * kQb + j];
        d += part[(4 + k) * kQb + j];
        cu += part[(8 + k) * kQb + j];
      }
      dc = r - dts[j] * cu;
      dd = d + cu;
    };
    // the per-warp sums: <dH, H> (five warps), sum_j w_j v_j and dD (sixteen)
    const float* ws = wsum + hh * 48;
    float s_hd = lane < 5 ? ws[lane] : 0.f, s_wv = lane < 16 ? ws[16 + lane] : 0.f;
    float s_dd = lane < 16 ? ws[32 + lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s_hd += __shfl_xor_sync(0xffffffffu, s_hd, o);
      s_wv += __shfl_xor_sync(0xffffffffu, s_wv, o);
      s_dd += __shfl_xor_sync(0xffffffffu, s_dd, o);
    }
    const float extra = tc::fast_exp2(hsum[4 * hh]) * s_hd + s_wv;
    const int j1 = kQb - 1 - 2 * lane, j2 = j1 - 1;  // lane l: entries 63 - 2l, 62 - 2l
    float dc1, dd1, dc2, dd2;
    sums(j1, dc1, dd1);
    sums(j2, dc2, dd2);
    const float a1 = dc1 + (j1 == len - 1 ? extra : 0.f);
    const float a2 = dc2 + (j2 == len - 1 ? extra : 0.f);
    if (lane == 0 && p.dD) atomicAdd(p.dD + h, s_dd);
    float v = a1 + a2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    const float r2 = v, r1 = v - a2;
    const float Ah = p.A[h];
    float da = 0.f;
    if (j1 < len) {
      p.ddt[(k.tok0 + j1) * p.H + h] = dd1 + Ah * r1;
      da = fmaf(dts[j1], r1, da);
    }
    if (j2 < len) {
      p.ddt[(k.tok0 + j2) * p.H + h] = dd2 + Ah * r2;
      da = fmaf(dts[j2], r2, da);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
    if (lane == 0) atomicAdd(p.dA + h, da);
  }
  // ---- dB, dC of the slice's heads: warp w, dstate rows 32 (w % 4) + lane,
  //      tokens 16 (w / 4).. (columns j and 64 + j summed)
  if (math) {
    float c0[16], c1[16], b0[16], b1[16];
    tc::tmem_ld16(tm + lanebase + cDC + c16, c0);
    tc::tmem_ld16(tm + lanebase + cDC + 64 + c16, c1);
    tc::tmem_ld16(tm + lanebase + cDB + c16, b0);
    tc::tmem_ld16(tm + lanebase + cDB + 64 + c16, b1);
    tc::tmem_ld_wait();
    tc::tie16(c0);
    tc::tie16(c1);
    tc::tie16(b0);
    tc::tie16(b1);
    const int n = 32 * qd + lane;
    if (n < N) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = c16 + e;
        if (j < len) {
          const long long row = ((k.tok0 + j) * p.G + g) * N + n;
          atomicAdd(p.dC + row, c0[e] + c1[e]);
          atomicAdd(p.dB + row, b0[e] + b1[e]);
        }
      }
    }
  }
  if (!ok && p.status) atomicCAS(p.status, 0, (int)SSD_ERR_TIMEOUT);
  // the last H, dH loads complete before the block's shared memory goes
  // (they all did unless a wait expired; bounded)
  if (!math && lane == 0 && hd_issued > 0)
    (void)tc::mbar_wait(hdbar, (uint32_t)((hd_issued - 1) & 1), p.wait_polls);
  tc::tc_fence_before();
  __syncthreads();
  if (!math) {  // every MMA of the block complete before its tensor memory is freed
    if (tc::elect_one()) tc::mma_commit(&bars[5]);
    __syncwarp();
    tc::mbar_wait(&bars[5], 0);
    tc::tmem_dealloc(tm, 512);
  }
}
#undef KD
#undef MD

// ---------------------------------------------------------------- state scans, tcgen05
// The states entering each chunk (forwards from init) and the adjoints
// leaving each chunk (backwards from dL/dfinal) for the tcgen05 gradient
// kernel: one block per (head, batch row, direction, half of headdim) walks
// the row's chunks in order with its 128 x 32 part of the state in
// registers, so every state is written once.  Storage is transposed and
// split for the gradient kernel's operands: bf16 hi/lo pairs (hi = rn(v), lo
// = rn(v - hi)), each [chunk][head][n][q] (dstate rows of headdim values), in
// the workspace of the fp32 states; dinit [batch][head][q][n] in fp32.  Per
// chunk the local sum
//   forwards:  sum_j B_j (w_j x_j)^T,       w_j = exp(cum_last - cum_j) dt_j
//   backwards: sum_i C_i (exp(cum_i) dy_i)^T
// over the block's 32 columns is one M = 128 (n) x N = 64 tcgen05 product
// over the chunk's 64 tokens: B^T (or C^T) read MN-major, times the weighted
// rows as [hi | lo] (32 columns each) in one MN-major tile; the state then
// becomes exp(cum_last) state + hi + lo.  Warps 0-3 hold the state (row n =
// TMEM lane n) and write it out through two 64B-swizzled shared tiles (hi,
// lo) with TMA stores; warps 4-7 convert the operands of a two-slot ring
// whose rows arrive by TMA; warp 8 issues those copies (a slot's next ones
// once its product has read it, with an L2 prefetch of the x or dy rows two
// steps further) and the MMAs into a double-buffered accumulator.  Three
// blocks fit on an SM.  Every wait is bounded (SSD_ERR_TIMEOUT).
namespace sc {
constexpr int kStages = 2;
constexpr int kQH = 32;                     // headdim columns per block (half of 64)
constexpr uint32_t kAtom = 8192;            // 64 rows x 128 bytes
constexpr uint32_t kSlotBytes = 3 * kAtom;  // U (64 tokens x [hi 32 | lo 32]), V (64 tokens x 128 n)
constexpr int kThreads = 32 * 9;
constexpr int kTabF = 144;  // floats per (chunk, head) of the weight table
constexpr uint32_t oTab = kStages * kSlotBytes;  // [2][64] the slots' row weights
constexpr uint32_t oStg = oTab + 1024;  // [2][128 rows][32 bf16] 64B-swizzled tiles: the state out (hi, lo)
constexpr uint32_t kStgHalf = 8192;
constexpr uint32_t oBar = oStg + 16384;  // full[2], empty[2], acc full[2], acc free[2], drain; TMEM base
constexpr uint32_t kSmem = oBar + 128 + 1024;
constexpr uint32_t kId = tc::idesc_bf16(128, 64, true, true);
}  // namespace sc

// The weight table of the tensor-core path, per (chunk, head): the forward
// weights w_j = exp(cum_last - cum_j) dt_j in [0, 64), the adjoint weights
// exp(cum_i) in [64, 128), exp(cum_last) at 128 (rows past the chunk's end
// have dt = 0).  One warp per head, lane l on rows 2l and 2l + 1.
__global__ void __launch_bounds__(256) bwd_tab_kernel(BP p) {
  const int c = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 8 + w;
  {  // the accumulated gradients start at zero (dB, dC in pairs: dstate is even)
    const long long ntok = (long long)(gridDim.x / p.nc) * p.T;
    const long long nth = (long long)gridDim.x * gridDim.y * blockDim.x;
    const long long i0 = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nbc = ntok * p.G * p.N / 2;
    for (long long i = i0; i < nbc; i += nth) {
      reinterpret_cast<float2*>(p.dB)[i] = make_float2(0.f, 0.f);
      reinterpret_cast<float2*>(p.dC)[i] = make_float2(0.f, 0.f);
    }
    for (long long i = i0; i < ntok * p.H; i += nth) p.ddt[i] = 0.f;
    if (i0 < p.H) {
      p.dA[i0] = 0.f;
      if (p.dD) p.dD[i0] = 0.f;
    }
  }
  if (h >= p.H) return;
  const Chunk k = chunk_of(p, c);
  const float Ah2 = p.A[h] * tg::kLog2e;
  const int j0 = 2 * lane, j1 = j0 + 1;
  const float d0 = j0 < k.len ? ldin<true>(p.dt, (k.tok0 + j0) * p.H + h) : 0.f;
  const float d1 = j1 < k.len ? ldin<true>(p.dt, (k.tok0 + j1) * p.H + h) : 0.f;
  const float a1 = d1 * Ah2;
  float sum = d0 * Ah2 + a1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, sum, o);
    if (lane >= o) sum += u;
  }
  const float cm1 = sum, cm0 = sum - a1;
  const float lst = __shfl_sync(0xffffffffu, ((k.len - 1) & 1) ? cm1 : cm0, (k.len - 1) >> 1);
  float* row = p.tab + ((long long)c * p.H + h) * sc::kTabF;
  row[j0] = tc::fast_exp2(lst - cm0) * d0;
  row[j1] = tc::fast_exp2(lst - cm1) * d1;
  row[64 + j0] = tc::fast_exp2(cm0);
  row[64 + j1] = tc::fast_exp2(cm1);
  if (lane == 0) row[128] = tc::fast_exp2(lst);
}

__global__ void __launch_bounds__(sc::kThreads, 3)
    bwd_scan_kernel(BP p, const __grid_constant__ CUtensorMap map_sth,
                    const __grid_constant__ CUtensorMap map_stl,
                    const __grid_constant__ CUtensorMap map_adh,
                    const __grid_constant__ CUtensorMap map_adl,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c,
                    const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_dy) {
  using namespace sc;
  using tc::f2;
  const int h = blockIdx.x, b = blockIdx.y, dir = blockIdx.z >> 1, qh = blockIdx.z & 1;
  const int P = p.P, N = p.N, nc = p.nc;
  const int q0 = kQH * qh;  // this block's headdim columns q0 .. q0 + 31
  if (q0 >= P) return;      // (the whole block: headdim <= 32 needs one half)
  extern __shared__ unsigned char ssm_raw[];
  const uint32_t raw_s = tc::smem_u32(ssm_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  unsigned char* base = ssm_raw + (sb - raw_s);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + oBar);
  uint32_t* tptr = reinterpret_cast<uint32_t*>(base + oBar + 80);  // bars[8]: the drain
  volatile int* abort_f = reinterpret_cast<volatile int*>(base + oBar + 84);
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int g = (int)((long long)h * p.G / p.H);
  bool ok = true;
  const auto chunk_at = [&](int s) { return b * nc + (dir == 0 ? s : nc - 1 - s); };
  const float* tabh = p.tab + (long long)h * kTabF;  // + chunk * H * kTabF

  if (w == 8) {
    if (lane == 0) {
      for (int i = 0; i < 2; ++i) tc::mbar_init(&bars[i], 128);  // full: converter threads
      for (int i = 2; i < 6; ++i) tc::mbar_init(&bars[i], 1);    // empty, acc full: MMA commits
      for (int i = 6; i < 8; ++i) tc::mbar_init(&bars[i], 128);  // acc free: state threads
      tc::mbar_init(&bars[8], 1);                                // drain of the last MMAs
      for (int i = 11; i < 13; ++i) tc::mbar_init(&bars[i], 1);  // copies landed (TMA)
      *abort_f = 0;
      tc::fence_mbar_init();
    }
    __syncwarp();
    tc::tmem_alloc(tptr, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tptr;

  // Step s arrives in slot s % 2 by TMA (B or C rows, x or dy rows, the row
  // weights; bars[11 + slot] count the bytes), issued by the MMA warp: steps
  // 0 and 1 at once, step s + 2 when the product of step s has completed.
  uint64_t* cfull = &bars[11];
  int issued = 0;  // MMA warp, lane 0: the steps whose copies it issued
  const auto issue = [&](int s) {
    const int sl = s % kStages;
    const Chunk k = chunk_of(p, chunk_at(s));
    unsigned char* st = base + sl * kSlotBytes;
    tc::mbar_arrive_expect_tx(&cfull[sl], 2 * kAtom + (dir == 0 ? kAtom / 2 : kAtom) + 256);
    const CUtensorMap* mv = dir == 0 ? &map_b : &map_c;  // [tokens][G][N]: 64 tokens x 64 n
    tc::tma_load_3d(st + kAtom, mv, &cfull[sl], 0, g, (int)k.tok0);
    tc::tma_load_3d(st + 2 * kAtom, mv, &cfull[sl], 64, g, (int)k.tok0);
    // x (bf16) or dy (fp32), 32 columns of 64 tokens, row j at 64 j (x) or 128 j (dy)
    tc::tma_load_3d(st, dir == 0 ? &map_x : &map_dy, &cfull[sl], q0, h, (int)k.tok0);
    tc::bulk_load(base + oTab + 256 * sl, tabh + (long long)chunk_at(s) * p.H * kTabF + 64 * dir,
                  256, &cfull[sl]);
    if (s + 2 < nc) {  // the x or dy rows of two steps later into L2 (B and C rows are there)
      const Chunk kp = chunk_of(p, chunk_at(s + 2));
      tc::tma_prefetch_3d(dir == 0 ? &map_x : &map_dy, q0, h, (int)kp.tok0);
    }
  };
  // a slot's earlier copies complete (bounded) before it is refilled, so that
  // the phases of its barrier never overlap, even after an expired wait
  const auto issue_next = [&](int s) {
    if (issued != s) return;
    if (s >= kStages && !tc::mbar_wait(&cfull[s % kStages], ((s / kStages) - 1) & 1, p.wait_polls))
      return;
    issue(s);
    issued = s + 1;
  };
  if (w >= 4 && w < 8) {
    // ---- converters: step s has arrived in slot s % 2 by TMA; w o x (or
    //      exp(cum) o dy) for the block's 32 columns as [hi | lo] in one tile
    const int ct = t - 128;
    for (int s = 0; s < nc; ++s) {
      const int slot = s % kStages;
      ok &= bwait(&cfull[slot], (s / kStages) & 1, abort_f, p.wait_polls);
      const int len = chunk_of(p, chunk_at(s)).len;
      const float* wrow = reinterpret_cast<const float*>(base + oTab + 256 * slot);
      unsigned char* st = base + slot * kSlotBytes;
      if (len < kQb) {  // rows past a short chunk's end (the next tokens' B or C) read as zero
        for (int e = ct; e < (kQb - len) * 16; e += 128) {
          const int j = len + (e >> 4), c = e & 15;
          *reinterpret_cast<uint4*>(st + kAtom + (c >> 3) * kAtom + 128 * j + 16 * (c & 7)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      if (dir == 0) {
        uint4 xr[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int e = ct + 128 * r, j = e >> 2, q8 = (e & 3) * 8;
          xr[r] = *reinterpret_cast<const uint4*>(st + 64 * j + 2 * q8);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the raw rows are read before the tile overwrites them
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int e = ct + 128 * r, j = e >> 2, q8 = (e & 3) * 8;
          const float wj = j < len ? wrow[j] : 0.f;
          const uint4 xv = xr[r];
          const f2 ww{wj, wj};
          const f2 v[4] = {tc::mul2(tc::bf2(xv.x), ww), tc::mul2(tc::bf2(xv.y), ww),
                           tc::mul2(tc::bf2(xv.z), ww), tc::mul2(tc::bf2(xv.w), ww)};
          uint4 hi, lo;
          tg::split8(v, hi, lo);
          if (j >= len) hi = lo = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(st + tg::swo(j, q8)) = hi;
          *reinterpret_cast<uint4*>(st + tg::swo(j, kQH + q8)) = lo;
        }
      } else {
        float4 raw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) raw[r] = *reinterpret_cast<const float4*>(st + 16 * (ct + 128 * r));
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the raw rows are read before the tile overwrites them
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int e = ct + 128 * r, j = e >> 3, q4 = (e & 7) * 4;
          const float wj = wrow[j];
          float4 v = raw[r];
          if (j < len) {
            v.x *= wj;
            v.y *= wj;
            v.z *= wj;
            v.w *= wj;
          } else {
            v = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          tg::split4_at(st + tg::swo(j, q4), st + tg::swo(j, kQH + q4), v);
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars[slot]);
    }
  } else if (w == 8) {
    // ---- MMA warp
    if (lane == 0)
      for (int s = 0; s < kStages && s < nc; ++s) issue_next(s);
    for (int s = 0; s < nc; ++s) {
      const int slot = s % kStages, a = s & 1;
      ok &= bwait(&bars[slot], (s / kStages) & 1, abort_f, p.wait_polls);
      if (s >= 2) ok &= bwait(&bars[6 + a], ((s >> 1) - 1) & 1, abort_f, p.wait_polls);
      tc::tc_fence_after();
      if (tc::elect_one()) {
        const uint32_t s0 = sb + slot * kSlotBytes;
        const uint64_t dv = tc::sdesc_sw128(s0 + kAtom, kAtom, 1024);  // V^T, MN-major
        const uint64_t du = tc::sdesc_sw128(s0, kAtom, 1024);          // [U hi | U lo], MN-major
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tm + 64 * a, dv + kk * 128, du + kk * 128, kId, kk > 0);
        tc::mma_commit(&bars[2 + slot]);
        if (!(p.hold == 2 && s == 0 && h == 0 && b == 0 && dir == 0 && qh == 0))
          tc::mma_commit(&bars[4 + a]);  // (the test hook holds back the first one of one block)
      }
      __syncwarp();
      // the slot's next copies, once this product has read it (bounded)
      if (lane == 0 && s + kStages < nc &&
          tc::mbar_wait(&bars[2 + slot], (uint32_t)((s / kStages) & 1), p.wait_polls))
        issue_next(s + kStages);
      __syncwarp();
    }
    // every MMA of the block complete before its tensor memory is freed, and
    // the last copies landed before its shared memory goes (bounded)
    if (tc::elect_one()) tc::mma_commit(&bars[8]);
    __syncwarp();
    tc::mbar_wait(&bars[8], 0);
    if (lane == 0)
      for (int s = max(0, issued - kStages); s < issued; ++s)
        (void)tc::mbar_wait(&cfull[s % kStages], (s / kStages) & 1, p.wait_polls);
  } else {
    // ---- state warps: row n of the transposed state, the block's 32 columns
    const int n = 32 * w + lane;
    const uint32_t lb = (uint32_t)(32 * w) << 16;
    float S[kQH];
    const float* s0 = dir == 0 ? p.init : p.dfinal;
#pragma unroll
    for (int q = 0; q < kQH; ++q)
      S[q] = (s0 && q0 + q < P && n < N) ? s0[(((long long)b * p.H + h) * P + q0 + q) * N + n] : 0.f;
    // the chunks' decays, loaded four steps ahead
    float dcur[4], dnext[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) dcur[i] = i < nc ? tabh[(long long)chunk_at(i) * p.H * kTabF + 128] : 1.f;
    for (int s0i = 0; s0i < nc; s0i += 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dnext[i] = s0i + 4 + i < nc ? tabh[(long long)chunk_at(s0i + 4 + i) * p.H * kTabF + 128] : 1.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = s0i + i;
        if (s >= nc) break;
        const int a = s & 1;
        const long long c = chunk_at(s);
        {  // S out as bf16 hi/lo pairs (the gradient kernel's operand split):
           // row n into two 64-byte-swizzled stage tiles, then two TMA stores
          unsigned char* stg = base + oStg;
          if (t == 0) tc::bulk_wait_read<0>();  // the previous step's stores have read the stage
          asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
          for (int cq = 0; cq < kQH / 8; ++cq) {
            const f2 v[4] = {f2{S[8 * cq], S[8 * cq + 1]}, f2{S[8 * cq + 2], S[8 * cq + 3]},
                             f2{S[8 * cq + 4], S[8 * cq + 5]}, f2{S[8 * cq + 6], S[8 * cq + 7]}};
            uint4 hi, lo;
            tg::split8(v, hi, lo);
            const uint32_t o = (uint32_t)n * 64u + ((uint32_t)(cq ^ ((n >> 1) & 3)) << 4);
            *reinterpret_cast<uint4*>(stg + o) = hi;
            *reinterpret_cast<uint4*>(stg + kStgHalf + o) = lo;
          }
          tc::fence_proxy_async_smem();
          asm volatile("bar.sync 2, 128;" ::: "memory");
          if (t == 0) {
            const int row = (int)((c * p.H + h) * N);
            tc::tma_store_2d(dir == 0 ? &map_sth : &map_adh, stg, q0, row);
            tc::tma_store_2d(dir == 0 ? &map_stl : &map_adl, stg + kStgHalf, q0, row);
            tc::bulk_commit();
          }
        }
        const float dec = dcur[i];
        ok &= bwait(&bars[4 + a], (s >> 1) & 1, abort_f, p.wait_polls);
        tc::tc_fence_after();
#pragma unroll
        for (int qb = 0; qb < kQH; qb += 8) {  // columns qb.. of the hi half, 32 + qb.. of the lo half
          float vh[8], vl[8];
          const uint32_t col = tm + lb + 64 * a + qb;
          tc::tmem_ld8(col, vh);
          tc::tmem_ld8(col + kQH, vl);
          tc::tmem_ld_wait();
          tc::tie8(vh);
          tc::tie8(vl);
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) S[qb + i2] = fmaf(dec, S[qb + i2], vh[i2] + vl[i2]);
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&bars[6 + a]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) dcur[i] = dnext[i];
    }
    if (t == 0) tc::bulk_wait<0>();  // the state stores are complete
    if (dir == 1 && p.dinit && n < N) {
#pragma unroll
      for (int q = 0; q < kQH; ++q)
        if (q0 + q < P) p.dinit[(((long long)b * p.H + h) * P + q0 + q) * N + n] = S[q];
    }
  }
  if (!ok && p.status) atomicCAS(p.status, 0, (int)SSD_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  if (w == 8) tc::tmem_dealloc(tm, 128);
}

}  // namespace

namespace {
// Test hook (ssd_test_set_backward_wait).
std::atomic<unsigned long long> g_bwd_polls{0};
std::atomic<int> g_bwd_hold{0};
}  // namespace

bool bwd_chunked_supported(int P, int N) {
  // the state passes move float4s
  return P >= 1 && P <= kPmax && N >= 1 && N <= kNmax && (P * N) % 4 == 0;
}

size_t bwd_chunked_workspace_bytes(int batch, int T, int H, int P, int N) {
  const long long nch = (long long)batch * ((T + kQb - 1) / kQb);
  return 2 * align256(sizeof(float) * (size_t)nch * H * P * N) +
         align256(sizeof(float) * (size_t)nch * H) + align256(sizeof(float) * (size_t)nch * H * 144);
}

ssd_status_t bwd_chunked(const BwdArgs& a) {
  BP p;
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
  p.status = a.dev_status;
  {
    const unsigned long long polls = g_bwd_polls.load(std::memory_order_relaxed);
    p.wait_polls = polls == 0 ? (1u << 22) : (unsigned)std::min<unsigned long long>(polls, 1u << 30);
    p.hold = g_bwd_hold.load(std::memory_order_relaxed);
  }
  p.T = a.seqlen;
  p.H = a.H;
  p.P = a.P;
  p.N = a.N;
  p.G = a.G;
  p.nc = (a.seqlen + kQb - 1) / kQb;
  const bool bf = a.dtype == SSD_DT_BF16;
  const auto al = [](const void* q, uintptr_t m) { return (reinterpret_cast<uintptr_t>(q) & m) == 0; };
  p.vec = a.P % 8 == 0 && a.N % 8 == 0 && al(a.x, 15) && al(a.B, 15) && al(a.C, 15) && al(a.dy, 15);
  const long long nch = (long long)a.batch * p.nc;
  char* ws = static_cast<char*>(a.ws);
  const size_t sbytes = align256(sizeof(float) * (size_t)nch * a.H * a.P * a.N);
  p.st = reinterpret_cast<float*>(ws);
  p.ad = reinterpret_cast<float*>(ws + sbytes);
  p.dec = reinterpret_cast<float*>(ws + 2 * sbytes);
  p.tab = reinterpret_cast<float*>(ws + 2 * sbytes + align256(sizeof(float) * (size_t)nch * a.H));
  const dim3 pgrid((unsigned)((a.P * a.N / 4 + kThr - 1) / kThr), a.H, a.batch);
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (cudaFuncSetAttribute(bwd_grad_kernel<true>, at, (int)kGradSmem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_grad_tc_kernel, at, (int)tg::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_scan_kernel, at, (int)sc::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_grad_kernel<false>, at, (int)kGradSmem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_outer_kernel<true, 0>, at, (int)outer_smem<true>()) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_outer_kernel<true, 1>, at, (int)outer_smem<true>()) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_outer_kernel<false, 0>, at, (int)outer_smem<false>()) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_outer_kernel<false, 1>, at, (int)outer_smem<false>()) != cudaSuccess)
      attr_err = cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;
  const int hpg = a.H / a.G;
  const dim3 ggrid((unsigned)nch, a.G, (unsigned)((hpg + kHS - 1) / kHS));
  // The tensor-core path (bf16 inputs, headdim and dstate multiples of 8; x,
  // B, C and dy move as 16-byte vectors, dx, dB and dC in pairs): the state
  // scans (transposed states) and the tcgen05 gradient kernel.
  const bool tcp = bf && a.P % 8 == 0 && a.N % 8 == 0 && al(a.x, 15) && al(a.B, 15) &&
                   al(a.C, 15) && al(a.dy, 15) && al(a.dx, 7) && al(a.dB, 7) && al(a.dC, 7) &&
                   al(a.dinit, 3);
  if (tcp) {
    // (the table kernel also zeroes dA, ddt, dD, dB and dC)
    bwd_tab_kernel<<<dim3((unsigned)nch, (unsigned)((a.H + 7) / 8)), 256, 0, a.stream>>>(p);
    // the transposed states as bf16 hi/lo pairs: stored by the scans (32
    // columns x N rows per step), loaded by the gradient kernel (64 x 64 tiles)
    const long long selems = nch * a.H * a.N * a.P, slabs = nch * a.H;
    p.sth = reinterpret_cast<__nv_bfloat16*>(p.st);
    p.stl = p.sth + selems;
    p.adh = reinterpret_cast<__nv_bfloat16*>(p.ad);
    p.adl = p.adh + selems;
    CUtensorMap ms[4], ml[4];
    __nv_bfloat16* const sp[4] = {p.sth, p.stl, p.adh, p.adl};
    for (int i = 0; i < 4; ++i)
      if (!tc_make_map_bf16_sw64(&ms[i], sp[i], slabs * a.N, a.P, a.N) ||
          !tc_make_map_bf16_slab_sw128(&ml[i], sp[i], slabs, a.N, a.P))
        return SSD_ERR_CUDA;
    // the scans' per-step operands: B or C rows of one group (64 tokens x 64 of
    // dstate, 128-byte swizzle), x or dy rows of one head (64 tokens x 32 of headdim)
    CUtensorMap mb, mc, mx, mdy;
    const long long ntok = (long long)a.batch * a.seqlen;
    if (!tc_make_map_3d(&mb, a.B, 2, a.N, a.G, ntok, 64, 1, 64, true) ||
        !tc_make_map_3d(&mc, a.C, 2, a.N, a.G, ntok, 64, 1, 64, true) ||
        !tc_make_map_3d(&mx, a.x, 2, a.P, a.H, ntok, 32, 1, 64, false) ||
        !tc_make_map_3d(&mdy, a.dy, 4, a.P, a.H, ntok, 32, 1, 64, false))
      return SSD_ERR_CUDA;
    bwd_scan_kernel<<<dim3((unsigned)a.H, (unsigned)a.batch, 4), sc::kThreads, sc::kSmem, a.stream>>>(
        p, ms[0], ms[1], ms[2], ms[3], mb, mc, mx, mdy);
    bwd_grad_tc_kernel<<<ggrid, tg::kThreads, tg::kSmem, a.stream>>>(p, ml[0], ml[1], ml[2], ml[3]);
    count_launches(3);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  if (bwd_zero_grads(a) != cudaSuccess) return SSD_ERR_CUDA;
  if (bf) {
    bwd_outer_kernel<true, 0><<<ggrid, kThr, outer_smem<true>(), a.stream>>>(p);
    bwd_outer_kernel<true, 1><<<ggrid, kThr, outer_smem<true>(), a.stream>>>(p);
  } else {
    bwd_outer_kernel<false, 0><<<ggrid, kThr, outer_smem<false>(), a.stream>>>(p);
    bwd_outer_kernel<false, 1><<<ggrid, kThr, outer_smem<false>(), a.stream>>>(p);
  }
  bwd_pass_kernel<true><<<pgrid, kThr, 0, a.stream>>>(p);
  bwd_pass_kernel<false><<<pgrid, kThr, 0, a.stream>>>(p);
  if (bf)
    bwd_grad_kernel<true><<<ggrid, kThr, kGradSmem, a.stream>>>(p);
  else
    bwd_grad_kernel<false><<<ggrid, kThr, kGradSmem, a.stream>>>(p);
  count_launches(5);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd

extern "C" void ssd_test_set_backward_wait(unsigned long long polls, int hold) {
  ssd::g_bwd_polls.store(polls, std::memory_order_relaxed);
  ssd::g_bwd_hold.store(hold, std::memory_order_relaxed);
}
