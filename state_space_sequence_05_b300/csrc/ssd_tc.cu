// ssd_tc.cu -- tcgen05 tensor-core SSD forward for bf16 inputs, headdim 64,
// dstate 128 (the Mamba-2 2.7B layer shape).
//
// What it computes is the SSD chunked algorithm ("Transformers are SSMs
// Review", sec. 3-2 (4)) with 128-token chunks, per (sequence, head):
//
//   cum_i      = sum_{k<=i} dt_k A_h                       (chunk-local)
//   G          = C B^T                         (128 x 128, K = dstate)
//   S[i,j]     = G[i,j] exp(cum_i - cum_j) dt_j  for j <= i, else 0
//   Y_diag     = S X                           (intra-chunk quadratic form)
//   S_c^T      = B^T (w o X),  w_j = exp(cum_last - cum_j) dt_j   (chunk state)
//   Y_off      = C H_{c-1}^T                   (off-diagonal, state in)
//   y          = Y_diag + exp(cum_i) Y_off + D_h x
//   H_c        = exp(cum_last) H_{c-1} + S_c   (state passing)
//
// Precision: x, B and C arrive in bf16 and are used as they are.  The three
// operands the kernel derives (S, w o X and H) are fp32 values; each is
// written as a pair of bf16 numbers hi = bf16(v), lo = bf16(v - hi) and both
// halves are multiplied into the same fp32 accumulator, so the products see
// about 16 mantissa bits instead of 8.  (A single bf16 rounding of these
// operands alone costs up to ~2.6e-2 of RMS(y) in max error.)
//
// The chunk length is fixed at 128 = the tcgen05 tile height M.  Any chunk
// size gives the same function up to rounding (the decomposition is an
// exact reordering of the recurrence), so every chunk_size the API accepts
// runs with 128-token blocks here.
//
// Design (one persistent CTA per SM, 320 threads):
//   warp 8     TMA producer: per tile loads C (2 x 16 KB), B (2 x 16 KB) and
//              x (16 KB) into a 2-stage ring with the 128-byte swizzle the
//              MMA descriptors expect; draws work units from a global ticket.
//   warp 9     MMA issuer (one thread): C B^T -> TMEM; B^T X' -> TMEM;
//              C H^T -> TMEM; S X -> TMEM with S read from TMEM.
//   warps 0-7  CUDA-core math (256 threads, row r = lane of TMEM, column
//              half hp): cumulative decay, decay weights, the masked S
//              (written as bf16 pairs over the C B^T accumulator), the
//              epilogue, and the fp32 state H (registers) with its bf16 copy
//              in shared memory for the next chunk's C H^T.
// A work unit is one (sequence, head); the state never leaves the SM
// between chunks.  Every inter-warp wait is an mbarrier wait bounded in
// time; on expiry the kernel records SSD_ERR_TIMEOUT and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kQ = 128;  // chunk tokens = MMA M
constexpr int kP = 64;   // headdim
constexpr int kN = 128;  // dstate
constexpr int kStages = 2;
constexpr int kMathWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

constexpr uint32_t kTile = 16384;                 // one 128 x 64 bf16 tile
constexpr uint32_t kStageBytes = 5 * kTile;       // C0 C1 B0 B1 X
constexpr uint32_t kOffXw = kStages * kStageBytes;  // w o X as bf16 hi, lo (2 x 16 KB)
constexpr uint32_t kOffHt = kOffXw + 2 * kTile;     // H^T as bf16 hi, lo (2 x 16 KB)
constexpr uint32_t kOffTabs = kOffHt + 2 * kTile;   // c2[128] dt[128] part[8]
constexpr uint32_t kOffInfo = kOffTabs + 4 * 272;
constexpr uint32_t kSmemUse = kOffInfo + 128;
constexpr uint32_t kSmemBytes = kSmemUse + 1024;  // slack for 1024-B alignment

// TMEM columns (fp32 accumulators, 128 lanes).
constexpr uint32_t kColCB = 0;     // 2 x 128: C B^T, overwritten by bf16 S hi (64) | lo (64)
constexpr uint32_t kColYD = 256;   // 64: S X
constexpr uint32_t kColST = 320;   // 64: chunk state (transposed: lane n, column p)
constexpr uint32_t kColYO = 384;   // 64: C H^T
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait

struct TileInfo {
  long long t0;  // first token of the chunk
  int s, h;      // sequence, head
  int len;       // valid rows (1..128); 0 = no more work
  int first, last;
  int pad;
};

struct Params {
  const __nv_bfloat16* dt;
  const float* A;
  const float* D;
  const float* init;
  float* y;
  float* final_states;
  SeqInfo si;
  const int32_t* offs;  // plan; offs[nseq+1] != 0 => malformed cu_seqlens
  int* ticket;
  int32_t* status;
  int H, G, nunits;
};

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait: polls until `parity` completes or kWaitNs passes.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = gtime();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (gtime() - t0 > kWaitNs) return false;
  }
}

// All 8 math warps meet at `bar` (phase parity `par`); bounded.  The math
// warps synchronise only through mbarriers so that a timed-out warp can
// leave without stranding the others at a hardware barrier.
__device__ __forceinline__ bool math_sync(uint64_t* bar, uint32_t par) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  return wait_bar(bar, par);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// v ~= hi + lo with hi = bf16(v), lo = bf16(v - hi); packs two such pairs.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float ha = __low2float(h), hb = __high2float(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf2(a - ha, b - hb);
}

// Write 32 fp32 values (one row's half) as hi and lo bf16 rows in two
// 128B-swizzled tiles, 16-byte chunks 4*hp .. 4*hp+3 of row `row`.
__device__ __forceinline__ void store_split_row(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                                int hp, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 h4, l4;
    split2(v[8 * c + 0], v[8 * c + 1], h4.x, l4.x);
    split2(v[8 * c + 2], v[8 * c + 3], h4.y, l4.y);
    split2(v[8 * c + 4], v[8 * c + 5], h4.z, l4.z);
    split2(v[8 * c + 6], v[8 * c + 7], h4.w, l4.w);
    const uint32_t off = sw128_offset(row, 4 * hp + c);
    *reinterpret_cast<uint4*>(hi_tile + off) = h4;
    *reinterpret_cast<uint4*>(lo_tile + off) = l4;
  }
}

struct Smem {
  uint8_t* base;
  uint64_t* bars;
  __device__ uint8_t* stage(int s) const { return base + s * kStageBytes; }
  __device__ uint8_t* C(int s, int half) const { return stage(s) + half * kTile; }
  __device__ uint8_t* B(int s, int half) const { return stage(s) + (2 + half) * kTile; }
  __device__ uint8_t* X(int s) const { return stage(s) + 4 * kTile; }
  __device__ uint8_t* Xw(int part) const { return base + kOffXw + part * kTile; }
  __device__ uint8_t* Ht(int part) const { return base + kOffHt + part * kTile; }
  __device__ float* c2() const { return reinterpret_cast<float*>(base + kOffTabs); }
  __device__ float* dtt() const { return c2() + 128; }
  __device__ float* part() const { return c2() + 256; }
  __device__ TileInfo* info(int s) const {
    return reinterpret_cast<TileInfo*>(base + kOffInfo) + s;
  }
};

// barrier indices
enum {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1, kCbFull0, kCbFull1, kCbsEmpty0, kCbsEmpty1,
  kXsReady, kSReady, kHReady, kAccFull, kAccEmpty, kSync0, kSync1, kSync2, kMmaDone,
  kNumBars
};

__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_fwd_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_c, Params prm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  Smem sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  sm.bars = bars;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars[kFull0], 1);
    mbar_init(&bars[kFull1], 1);
    mbar_init(&bars[kEmpty0], 1 + kMathWarps);
    mbar_init(&bars[kEmpty1], 1 + kMathWarps);
    mbar_init(&bars[kCbFull0], 1);
    mbar_init(&bars[kCbFull1], 1);
    mbar_init(&bars[kCbsEmpty0], 1);
    mbar_init(&bars[kCbsEmpty1], 1);
    mbar_init(&bars[kXsReady], kMathWarps);
    mbar_init(&bars[kSReady], kMathWarps);
    mbar_init(&bars[kHReady], kMathWarps);
    mbar_init(&bars[kAccFull], 1);
    mbar_init(&bars[kAccEmpty], kMathWarps);
    mbar_init(&bars[kSync0], kMathWarps);
    mbar_init(&bars[kSync1], kMathWarps);
    mbar_init(&bars[kSync2], kMathWarps);
    mbar_init(&bars[kMmaDone], 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  auto fail = [&](int code) {
    report(prm.status, code);
    atomicExch(&abort_sh, 1);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map_x);
      prefetch_tmap(&map_b);
      prefetch_tmap(&map_c);
      const bool plan_ok = prm.offs[prm.si.nseq + 1] == 0;
      uint32_t it = 0;
      bool ok = true;
      while (ok && plan_ok) {
        const int u = atomicAdd(prm.ticket, 1);
        if (u >= prm.nunits) break;
        const int s = u / prm.H, h = u % prm.H;
        const int g = (int)((long long)h * prm.G / prm.H);
        const long long b = prm.si.begin(s), e = prm.si.end(s);
        const int ntiles = (int)((e - b + kQ - 1) / kQ);
        for (int t = 0; t < ntiles; ++t, ++it) {
          const int st = it & 1;
          if (it >= 2 && !wait_bar(&bars[kEmpty0 + st], ((it >> 1) - 1) & 1)) {
            fail(SSD_ERR_TIMEOUT);
            ok = false;
            break;
          }
          if (*(volatile int*)&abort_sh) { ok = false; break; }
          TileInfo* inf = sm.info(st);
          inf->t0 = b + (long long)t * kQ;
          inf->s = s;
          inf->h = h;
          inf->len = (int)min((long long)kQ, e - inf->t0);
          inf->first = t == 0;
          inf->last = t == ntiles - 1;
          const int row = (int)inf->t0;
          mbar_arrive_expect_tx(&bars[kFull0 + st], kStageBytes);
          tma_load_2d(sm.C(st, 0), &map_c, &bars[kFull0 + st], g * kN, row);
          tma_load_2d(sm.C(st, 1), &map_c, &bars[kFull0 + st], g * kN + 64, row);
          tma_load_2d(sm.B(st, 0), &map_b, &bars[kFull0 + st], g * kN, row);
          tma_load_2d(sm.B(st, 1), &map_b, &bars[kFull0 + st], g * kN + 64, row);
          tma_load_2d(sm.X(st), &map_x, &bars[kFull0 + st], h * kP, row);
        }
      }
      // sentinel: no more work
      const int st = it & 1;
      if (ok && (it < 2 || wait_bar(&bars[kEmpty0 + st], ((it >> 1) - 1) & 1))) {
        sm.info(st)->len = 0;
        mbar_arrive(&bars[kFull0 + st]);
      } else {
        if (ok) fail(SSD_ERR_TIMEOUT);
        // aborting: loads still in flight must land before the CTA may exit
        for (uint32_t k = (it >= 2 ? it - 2 : 0); k < it; ++k)
          (void)wait_bar(&bars[kFull0 + (k & 1)], (k >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idCB = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idST = idesc_bf16(128, 64, true, true);
      constexpr uint32_t idYO = idesc_bf16(128, 64, false, true);
      constexpr uint32_t idYD = idesc_bf16(128, 64, false, true);
      uint32_t it = 0;
      bool issued = false;
      while (true) {
        const int st = it & 1;
        if (!wait_bar(&bars[kFull0 + st], (it >> 1) & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        if (sm.info(st)->len == 0 || *(volatile int*)&abort_sh) break;
        const uint32_t cbcol = tmem + kColCB + st * 128;
        if (it >= 2 && !wait_bar(&bars[kCbsEmpty0 + st], ((it >> 1) - 1) & 1)) {
          fail(SSD_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t aC0 = smem_u32(sm.C(st, 0)), aC1 = smem_u32(sm.C(st, 1));
        const uint32_t aB0 = smem_u32(sm.B(st, 0)), aB1 = smem_u32(sm.B(st, 1));
        const uint32_t aX = smem_u32(sm.X(st));
        // G = C B^T (both K-major; K = dstate over two 64-wide boxes)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = (k & 3) * 32;
          mma_bf16(cbcol, sdesc_sw128((k < 4 ? aC0 : aC1) + kb, 16, 1024),
                   sdesc_sw128((k < 4 ? aB0 : aB1) + kb, 16, 1024), idCB, k > 0);
        }
        mma_commit(&bars[kCbFull0 + st]);
        issued = true;
        if (it >= 1 && !wait_bar(&bars[kAccEmpty], (it - 1) & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        if (!wait_bar(&bars[kXsReady], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        // chunk state S_c^T (n x p) = B^T (w o X): A MN-major (B rows j), B MN-major
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t aXw = smem_u32(sm.Xw(part));
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(tmem + kColST, sdesc_sw128(aB0 + k * 2048, kTile, 1024),
                     sdesc_sw128(aXw + k * 2048, kTile, 1024), idST, part > 0 || k > 0);
        }
        if (!wait_bar(&bars[kHReady], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        // Y_off = C H^T: A K-major (C), B MN-major (H^T rows n)
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t aH = smem_u32(sm.Ht(part));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t kb = (k & 3) * 32;
            mma_bf16(tmem + kColYO, sdesc_sw128((k < 4 ? aC0 : aC1) + kb, 16, 1024),
                     sdesc_sw128(aH + k * 2048, kTile, 1024), idYO, part > 0 || k > 0);
          }
        }
        if (!wait_bar(&bars[kSReady], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        // Y_diag = S X, S (bf16 pairs) read from TMEM
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16_tmem_a(tmem + kColYD, cbcol + part * 64 + k * 8,
                            sdesc_sw128(aX + k * 2048, kTile, 1024), idYD, part > 0 || k > 0);
        mma_commit(&bars[kAccFull]);
        mma_commit(&bars[kEmpty0 + st]);
        mma_commit(&bars[kCbsEmpty0 + st]);
        ++it;
      }
      if (issued) {
        // every MMA issued must complete before TMEM is released
        mma_commit(&bars[kMmaDone]);
        if (!wait_bar(&bars[kMmaDone], 0)) fail(SSD_ERR_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ math warps
    const int r = tid & 127;       // TMEM lane: token row i / state row n / token j
    const int hp = tid >> 7;       // column half
    const int wq = warp & 3;       // lane quarter of this warp
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    float hreg[32];                // H[p][n = r] for p = 32 hp + q
#pragma unroll
    for (int q = 0; q < 32; ++q) hreg[q] = 0.f;
    uint32_t it = 0;
    while (true) {
      const int st = it & 1;
      if (!wait_bar(&bars[kFull0 + st], (it >> 1) & 1)) { fail(SSD_ERR_TIMEOUT); break; }
      const TileInfo inf = *sm.info(st);
      if (inf.len == 0 || *(volatile int*)&abort_sh) break;
      const int h = inf.h;
      const float A2 = prm.A[h] * kLog2e;
      const float Dh = prm.D ? prm.D[h] : 0.f;
      // -- unit start: load the initial state
      if (inf.first) {
        const float* ini = prm.init ? prm.init + ((long long)inf.s * prm.H + h) * (kP * kN)
                                    : nullptr;
#pragma unroll
        for (int q = 0; q < 32; ++q)
          hreg[q] = ini ? __ldg(ini + (32 * hp + q) * kN + r) : 0.f;
        store_split_row(sm.Ht(0), sm.Ht(1), r, hp, hreg);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kHReady]);
      }
      // -- cumulative decay (log2 domain) over the chunk
      float* c2 = sm.c2();
      float* dtt = sm.dtt();
      float* part = sm.part();
      float d = 0.f, v = 0.f;
      if (hp == 0) {
        if (r < inf.len) d = __bfloat162float(prm.dt[(inf.t0 + r) * prm.H + h]);
        v = d * A2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += t;
        }
        if (lane == 31) part[wq] = v;
      }
      if (!math_sync(&bars[kSync0], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
      if (hp == 0) {
        float off = 0.f;
        for (int w = 0; w < wq; ++w) off += part[w];
        c2[r] = v + off;
        dtt[r] = d;
      }
      if (!math_sync(&bars[kSync1], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
      const float c2_last = c2[kQ - 1];
      const float c2_r = c2[r];
      const float dt_r = dtt[r];
      // -- X' = w o X (row j = r, p chunks 4hp .. 4hp+3)
      {
        const float w = exp2f(c2_last - c2_r) * dt_r;
        const uint8_t* Xs = sm.X(st);
        float xw[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 xv = *reinterpret_cast<const uint4*>(Xs + sw128_offset(r, 4 * hp + c));
          xw[8 * c + 0] = w * bf_lo(xv.x);
          xw[8 * c + 1] = w * bf_hi(xv.x);
          xw[8 * c + 2] = w * bf_lo(xv.y);
          xw[8 * c + 3] = w * bf_hi(xv.y);
          xw[8 * c + 4] = w * bf_lo(xv.z);
          xw[8 * c + 5] = w * bf_hi(xv.z);
          xw[8 * c + 6] = w * bf_lo(xv.w);
          xw[8 * c + 7] = w * bf_hi(xv.w);
        }
        store_split_row(sm.Xw(0), sm.Xw(1), r, hp, xw);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kXsReady]);
      }
      // -- S = (C B^T) o exp(cum_i - cum_j) dt_j, causal, written over C B^T
      {
        if (!wait_bar(&bars[kCbFull0 + st], (it >> 1) & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        const uint32_t cbcol = tmem + kColCB + st * 128 + lane_addr;
        const int i = r;
        const int jbase = 64 * hp;
        uint32_t pkh[32], pkl[32];   // S hi / lo, bf16 pairs, columns jbase .. jbase+63
        // this warp's rows are 32 wq .. 32 wq + 31; columns beyond them are 0
        const bool any = jbase <= 32 * wq + 31;
        if (any) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float g[32];
            tmem_ld32(cbcol + jbase + 32 * half, g);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int j0 = jbase + 32 * half + 2 * q, j1 = j0 + 1;
              const float s0 = j0 <= i ? g[2 * q] * exp2f(c2_r - c2[j0]) * dtt[j0] : 0.f;
              const float s1 = j1 <= i ? g[2 * q + 1] * exp2f(c2_r - c2[j1]) * dtt[j1] : 0.f;
              split2(s0, s1, pkh[16 * half + q], pkl[16 * half + q]);
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) pkh[q] = pkl[q] = 0u;
        }
        // every C B^T read of this chunk is done before any S write lands
        tc_fence_before();
        if (!math_sync(&bars[kSync2], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        const uint32_t scol = tmem + kColCB + st * 128 + lane_addr + 32 * hp;
        uint32_t tmp[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) tmp[q] = pkh[q];
        tmem_st16(scol, tmp);
#pragma unroll
        for (int q = 0; q < 16; ++q) tmp[q] = pkh[16 + q];
        tmem_st16(scol + 16, tmp);
#pragma unroll
        for (int q = 0; q < 16; ++q) tmp[q] = pkl[q];
        tmem_st16(scol + 64, tmp);
#pragma unroll
        for (int q = 0; q < 16; ++q) tmp[q] = pkl[16 + q];
        tmem_st16(scol + 64 + 16, tmp);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSReady]);
      }
      // -- epilogue and state update
      {
        if (!wait_bar(&bars[kAccFull], it & 1)) { fail(SSD_ERR_TIMEOUT); break; }
        tc_fence_after();
        float yd[32], yo[32], sv[32];
        tmem_ld32(tmem + kColYD + lane_addr + 32 * hp, yd);
        tmem_ld32(tmem + kColYO + lane_addr + 32 * hp, yo);
        tmem_ld32(tmem + kColST + lane_addr + 32 * hp, sv);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kAccEmpty]);
        // y row i = r
        if (r < inf.len) {
          const float ei = exp2f(c2_r);
          const uint8_t* Xs = sm.X(st);
          float* yrow = prm.y + ((inf.t0 + r) * prm.H + h) * kP + 32 * hp;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 xv = *reinterpret_cast<const uint4*>(Xs + sw128_offset(r, 4 * hp + c));
            const float xs[8] = {bf_lo(xv.x), bf_hi(xv.x), bf_lo(xv.y), bf_hi(xv.y),
                                 bf_lo(xv.z), bf_hi(xv.z), bf_lo(xv.w), bf_hi(xv.w)};
            float4 o0, o1;
            o0.x = yd[8 * c + 0] + ei * yo[8 * c + 0] + Dh * xs[0];
            o0.y = yd[8 * c + 1] + ei * yo[8 * c + 1] + Dh * xs[1];
            o0.z = yd[8 * c + 2] + ei * yo[8 * c + 2] + Dh * xs[2];
            o0.w = yd[8 * c + 3] + ei * yo[8 * c + 3] + Dh * xs[3];
            o1.x = yd[8 * c + 4] + ei * yo[8 * c + 4] + Dh * xs[4];
            o1.y = yd[8 * c + 5] + ei * yo[8 * c + 5] + Dh * xs[5];
            o1.z = yd[8 * c + 6] + ei * yo[8 * c + 6] + Dh * xs[6];
            o1.w = yd[8 * c + 7] + ei * yo[8 * c + 7] + Dh * xs[7];
            __stcs(reinterpret_cast<float4*>(yrow + 8 * c), o0);
            __stcs(reinterpret_cast<float4*>(yrow + 8 * c + 4), o1);
          }
        }
        // state: H_c[p][n=r] = exp(cum_last) H_{c-1} + S_c
        const float a = exp2f(c2_last);
#pragma unroll
        for (int q = 0; q < 32; ++q) hreg[q] = a * hreg[q] + sv[q];
        if (!inf.last) {
          store_split_row(sm.Ht(0), sm.Ht(1), r, hp, hreg);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kHReady]);
        } else if (prm.final_states) {
          float* fin = prm.final_states + ((long long)inf.s * prm.H + h) * (kP * kN);
#pragma unroll
          for (int q = 0; q < 32; ++q) fin[(32 * hp + q) * kN + r] = hreg[q];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kEmpty0 + st]);
      }
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}

// --------------------------------------------------------------------------
// host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a [rows, cols] row-major matrix, 64 x 128 boxes, 128B swizzle.
bool make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  });
  return n > 0 ? n : 148;
}

}  // namespace

bool tc_supported(const FwdArgs& a) {
  return a.dtype == SSD_DT_BF16 && a.P == kP && a.N == kN;
}

size_t tc_workspace_bytes(const FwdArgs& a) { return plan_bytes(a.nseq) + 256; }

ssd_status_t tc_forward(const FwdArgs& a) {
  char* ws = static_cast<char*>(a.ws);
  int32_t* offs = reinterpret_cast<int32_t*>(ws);
  int* ticket = reinterpret_cast<int*>(ws + plan_bytes(a.nseq));
  const long long ntok = (long long)a.batch * a.seqlen;
  cudaError_t err = launch_plan(a.cu, a.seqlen, (int)ntok, a.nseq, kQ, offs, a.dev_status,
                                a.stream, ticket, a.init, a.final_states, a.H, kP * kN);
  if (err != cudaSuccess) return SSD_ERR_CUDA;
  if (ntok == 0) return SSD_OK;
  CUtensorMap mx, mb, mc;
  if (!make_map(&mx, a.x, ntok, (long long)a.H * kP) ||
      !make_map(&mb, a.B, ntok, (long long)a.G * kN) ||
      !make_map(&mc, a.C, ntok, (long long)a.G * kN))
    return SSD_ERR_CUDA;
  Params p;
  p.dt = static_cast<const __nv_bfloat16*>(a.dt);
  p.A = a.A;
  p.D = a.D;
  p.init = a.init;
  p.y = a.y;
  p.final_states = a.final_states;
  p.si = SeqInfo{a.cu, a.seqlen, a.nseq};
  p.offs = offs;
  p.ticket = ticket;
  p.status = a.dev_status;
  p.H = a.H;
  p.G = a.G;
  p.nunits = a.nseq * a.H;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(ssd_tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;
  const int grid = p.nunits < sm_count() ? p.nunits : sm_count();
  if (grid <= 0) return SSD_OK;
  ssd_tc_fwd_kernel<<<grid, kThreads, kSmemBytes, a.stream>>>(mx, mb, mc, p);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
