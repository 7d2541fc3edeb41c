// ssd_tc2.cu -- tcgen05 tensor-core SSD forward for bf16 inputs, headdim 64,
// dstate 128 (the Mamba-2 2.7B layer shape), pipelined for throughput.
//
// It evaluates the SSD chunked algorithm ("Transformers are SSMs Review",
// sec. 3-2 (4)) with 128-token chunks.  Per (sequence, head) and chunk, with
// cum_i = sum_{k<=i} dt_k A_h (chunk-local) and the row factor
// f_i = exp(max(cum_i, -60 ln 2)):
//
//   G        = C B^T                                  (128 x 128, K = dstate)
//   S'[i,j]  = G[i,j] exp(cum_i - cum_j) dt_j / f_i   for j <= i, else 0
//              (+ D_h / f_i on the diagonal: the skip term D x)
//   S_c      = B^T (w o X),  w_j = exp(cum_last - cum_j) dt_j   (chunk state)
//   H_c      = exp(cum_last) H_{c-1} + S_c                      (state passing)
//   y_i      = f_i (S' X + C H_{c-1}^T)_i
//
// so the intra-chunk quadratic form and the off-diagonal term C state decay
// share one accumulator.  For a row whose decay from the chunk start is
// above 2^-60, f_i = exp(cum_i) and S'[i,j] = G[i,j] E_j with the per-chunk
// table E_j = exp(-cum_j) dt_j, which stays below 2^60 dt_j for every j <= i.
// A row decayed below 2^-60 takes f_i = 2^-60 and its own exponentials; the
// state term of such a row is then scaled by 2^-60 instead of its exact
// factor exp(cum_i) < 2^-60, an absolute change below 2^-60 |C_i H^T|.
//
// Precision: x, B and C are bf16 and used as they are.  The derived fp32
// operands S', w o X and H are each split into bf16 hi (v truncated) and lo
// ((v - hi) truncated), |v - hi - lo| < 2^-14 |v|; both halves are
// multiplied into fp32 accumulators (a single bf16 rounding of any of them
// costs 2-4e-2 of RMS(y) in max error on the 2.7B layer).  The hi and lo
// halves of w o X and of H are the two 64-column halves of one N = 128
// operand, so each K step is one 128 x 128 x 16 product.
//
// Work partition.  Each sequence is cut into segments of 4-12 chunks; a work
// unit is one (sequence, segment, head), handed out in that order by a global
// ticket, so a unit's predecessor (same sequence and head, previous segment)
// was taken earlier by a running CTA.  A unit
//   A. computes each chunk's state S_c on the tensor core, chunks walked
//      backwards, keeps it in a per-CTA scratch in global memory (L2-
//      resident: every thread reloads only what it stored, and drops the
//      lines from L2 unwritten once consumed) and folds it into the segment-
//      local end state H_loc;
//   H. takes the state entering the segment, H_in, from the initial state or
//      from its predecessor's published end state, and publishes its own,
//      exp(sum of the segment's dt A) H_in + H_loc, behind a release flag:
//      the composition of affine maps (a2, b2) o (a1, b1) = (a2 a1,
//      a2 b1 + b2) ("Mamba ... review", feghi.github.io, sec. 4) at segment
//      granularity;
//   B. runs the forward over its chunks from H_in with the kept chunk states.
//
// Shared memory holds two rings that turn over at different rates: C/B slots
// (a chunk's C and B tiles; in the segment-state pass the C half holds the
// chunk's w o X instead) are handed back once the chunk's C B^T and C H^T
// products have read them -- early, since the state chain needs no
// product of the forward pass -- and x slots (with the chunk's decay
// tables) once its S' X product has.
//
// Roles (one persistent CTA per SM, 608 threads):
//   warp 16    producer: TMA loads of C, B, x tiles (128-byte swizzle) and
//              the chunk's decay tables.
//   warp 17    MMA issuer (the whole warp; one elected lane issues): the
//              chunk-state products, C H^T and S' X.
//   warp 18    C B^T issuer: each forward chunk's C B^T as soon as its tiles
//              land.
//   warps 0-15 CUDA-core math (tensor-memory lane quarter w % 4, column
//              quarter w / 4): w o X (bf16 hi/lo), the decay mask S' (in
//              place over G in tensor memory), the fp32 running state chain,
//              the epilogue.
// Every wait is bounded; on expiry the kernel records SSD_ERR_TIMEOUT and
// unwinds with all tensor memory freed.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "ssd_tc_host.h"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kQ = kTcChunk;  // 128 tokens per chunk = MMA M
constexpr int kP = 64;        // headdim
constexpr int kN = 128;       // dstate
constexpr int kPN = kP * kN;
constexpr int kMathWarps = 16;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kGWarp = 18;
constexpr int kThreads = 608;

constexpr uint32_t kTile = 16384;              // 128 rows x 128 bytes (bf16)
constexpr int kCB = 2;                         // C/B slots: C0 C1 B0 B1 (64 KB)
constexpr int kXS = 3;                         // x slots (16 KB) with decay tables
constexpr uint32_t kCBBytes = 4 * kTile;
constexpr uint32_t kOffX = kCB * kCBBytes;     // x slots
constexpr uint32_t kOffHt = kOffX + kXS * kTile;  // H^T, bf16 hi then lo
constexpr uint32_t kOffTabs = kOffHt + 2 * kTile; // per x slot: c2, E (fp32), dt (bf16)
constexpr uint32_t kTabBytes = 128 * 4 + 128 * 4 + 128 * 2;
constexpr uint32_t kOffInfo = kOffTabs + kXS * kTabBytes;
constexpr uint32_t kOffBars = kOffInfo + kXS * 64;
constexpr uint32_t kBarBytes = 32 * 8;
constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 16;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kOffTabs % 16 == 0 && kOffBars % 8 == 0, "alignment");

// Tensor memory columns (128 lanes x 512 columns of 32 bits).
//   S buffers (2 x 128): G = C B^T, overwritten in place by S' (hi/lo pairs).
//   accumulators (2 x 128): a chunk-state product [B^T (w o X)_hi |
//   B^T (w o X)_lo] (lane n, column p of each half) in the segment-state
//   pass, or a forward accumulator [C H_hi^T + S' X | C H_lo^T] (lane i,
//   column p of each half).
constexpr uint32_t kColS = 0;
constexpr uint32_t kColAcc = 256;
constexpr uint32_t kTmemCols = 512;
// Chunks per unit, at most (its chunk states are kept in the CTA's scratch).
constexpr int kStSlots = kTcSegMax > kTcSegVarlen ? kTcSegMax : kTcSegVarlen;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kDeep = -60.f;  // log2 of the smallest row factor

enum : int { kKindA = 0, kKindB = 1, kKindEnd = 2 };

struct TileInfo {
  long long t0;   // first token of the chunk
  int s, h, sigma, unit;
  int len;        // valid rows (1..128)
  int kind;       // kKindA (segment-state pass), kKindB (forward), kKindEnd
  int cnt;        // chunks of this kind in the unit
  int last_seg;   // the unit is its sequence's last segment
  int pad[2];
};
static_assert(sizeof(TileInfo) <= 64, "tile info slot");

struct Params {
  const __nv_bfloat16* dt;
  const float* A;
  const float* D;
  const float* init;
  float* y;
  float* final_states;
  SeqInfo si;
  const int32_t* uoff;  // [nseq + 2]: unit offsets per sequence, then plan status
  int* ticket;          // ticket[0]: work ticket; ticket[1]: line of the first expired wait
  int* flags;           // per unit: 1 once its segment end state is published
  float* slots;         // per unit: segment end state [P][N] fp32
  float* stbuf;         // per CTA: the current unit's chunk states, kStSlots x [P][N] fp32
  int32_t* status;
  int H, G, seg;
  int y_v8;             // y is 32-byte aligned: 32-byte stores
  unsigned long long wait_ns;  // bound on every wait
  int hold_unit;        // test hook: this unit never publishes its end state (-1: none)
};

// barrier indices
enum {
  kCbFull0 = 0, kCbFull1,             // C/B slot loaded (TMA)
  kCbEmpty0, kCbEmpty1,               // C/B slot read (producer's and MMA issuer's commits)
  kXFull0, kXFull1, kXFull2,          // x slot loaded (TMA) and its tables written
  kXEmpty0, kXEmpty1, kXEmpty2,       // x slot done with (math warps + MMA commit)
  kWxFull0, kWxFull1,                 // w o X written into C/B slot (segment-state pass)
  kGFull0, kGFull1,                   // C B^T in S buffer (producer's commit)
  kSFull0, kSFull1, kSFree0, kSFree1, // S' written (math) / S buffer read by S' X
  kHtFull, kHtFree,                   // H^T operand tiles
  kAccFull0, kAccFull1, kAccFree0, kAccFree1,
  kSync,                              // math-warp rendezvous
  kMmaDone,                           // both issuers' last products
  kNumBars
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

struct Smem {
  uint8_t* base;
  __device__ uint8_t* C(int cb, int half) const { return base + cb * kCBBytes + half * kTile; }
  __device__ uint8_t* B(int cb, int half) const { return base + cb * kCBBytes + (2 + half) * kTile; }
  // w o X of a segment-state chunk, hi then lo, in its slot's C half
  __device__ uint8_t* W(int cb) const { return base + cb * kCBBytes; }
  __device__ uint8_t* X(int xs) const { return base + kOffX + xs * kTile; }
  __device__ uint8_t* Ht() const { return base + kOffHt; }
  // cumulative log2-decay of the chunk in x slot xs: c2[j] = sum_{k<=j} dt_k A log2(e)
  __device__ float* c2(int xs) const {
    return reinterpret_cast<float*>(base + kOffTabs + xs * kTabBytes);
  }
  // E[j] = exp(-cum_j) dt_j (0 beyond the valid rows; may be inf where unused)
  __device__ float* E(int xs) const {
    return reinterpret_cast<float*>(base + kOffTabs + xs * kTabBytes + 512);
  }
  // dt of the chunk (0 beyond the valid rows)
  __device__ __nv_bfloat16* dt(int xs) const {
    return reinterpret_cast<__nv_bfloat16*>(base + kOffTabs + xs * kTabBytes + 1024);
  }
  __device__ TileInfo* info(int xs) const {
    return reinterpret_cast<TileInfo*>(base + kOffInfo) + xs;
  }
};

// Parity of the completion of use `u` of a barrier that completes once per use.
__device__ __forceinline__ uint32_t par_of(uint32_t u) { return u & 1u; }
// Ring position of chunk number `it`: the C/B slot it % 2 (use it / 2 of
// that slot's barriers), the x slot it % 3 (use it / 3).
__device__ __forceinline__ uint32_t cb_par(uint32_t it) { return (it >> 1) & 1u; }
__device__ __forceinline__ int x_slot(uint32_t it) { return (int)(it % 3u); }
__device__ __forceinline__ uint32_t x_par(uint32_t it) { return (it / 3u) & 1u; }
// For a pair of barriers alternating between two buffers: parity of use `u`
// on barrier (u & 1).
__device__ __forceinline__ uint32_t par2_of(uint32_t u) { return (u >> 1) & 1u; }

__global__ void __launch_bounds__(kThreads, 1)
    ssd_fwd2_kernel(const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c, Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (tid == 0) report(prm.status, SSD_ERR_UNSUPPORTED);
    return;
  }
  Smem sm;
  sm.base = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + kOffBars);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(smem_raw + kOffBars + kBarBytes);
  int* abort_p = reinterpret_cast<int*>(smem_raw + kOffBars + kBarBytes + 4);
  const unsigned long long wns = prm.wait_ns;

  if (tid == 0) {
    for (int b = 0; b < kCB; ++b) {
      mbar_init(&bars[kCbFull0 + b], 1);   // expect-tx arrival
      mbar_init(&bars[kCbEmpty0 + b], 2);  // producer (G product or plain) + MMA issuer
      mbar_init(&bars[kWxFull0 + b], kMathWarps);
      mbar_init(&bars[kGFull0 + b], 1);
      mbar_init(&bars[kSFull0 + b], kMathWarps);
      mbar_init(&bars[kSFree0 + b], 1);
      mbar_init(&bars[kAccFull0 + b], 1);
      mbar_init(&bars[kAccFree0 + b], kMathWarps);
    }
    for (int b = 0; b < kXS; ++b) {
      mbar_init(&bars[kXFull0 + b], 2);               // expect-tx arrival + tables written
      mbar_init(&bars[kXEmpty0 + b], kMathWarps + 1);  // math warps + MMA issuer
    }
    mbar_init(&bars[kHtFull], kMathWarps);
    mbar_init(&bars[kHtFree], 1);
    mbar_init(&bars[kSync], kMathWarps);
    mbar_init(&bars[kMmaDone], 2);
    *abort_p = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    tmem_alloc(tmem_base_p, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_p;
  volatile int* abort_v = abort_p;

  auto fail_at = [&](int code, int line) {
    report(prm.status, code);
    atomicCAS(prm.ticket + 1, 0, line);
    atomicExch(abort_p, 1);
  };
#define fail(code) fail_at((code), __LINE__)

  // the plan kernel's results (unit offsets, ticket, flags) are ready past
  // this point (a no-op when the launch was not programmatic)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nseq = prm.si.nseq;
  const int nunits = prm.uoff[nseq];
  const bool plan_ok = prm.uoff[nseq + 1] == 0;

  // C B^T: 128 x 128 x 128 from the slot's C and B tiles (both K-major).
  constexpr uint32_t idG = idesc_bf16(128, 128, false, false);
  // chunk states: B^T (MN-major, M = n) times [w o X hi | lo] (MN-major, N = 128).
  constexpr uint32_t idSt = idesc_bf16(128, 128, true, true);
  // forward: C (K-major) times [H_hi | H_lo]^T (MN-major, N = 128), then
  // S' (tensor memory) times X (MN-major, N = 64) into the first half.
  constexpr uint32_t idCH = idesc_bf16(128, 128, false, true);
  constexpr uint32_t idSX = idesc_bf16(128, 64, false, true);
  constexpr uint64_t kT16 = kTile >> 4;  // one tile, in descriptor address units

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Walks the chunks of each work unit (ticket): its segment-state chunks
    // (backwards), then its forward chunks.  Lane 0 issues the TMA loads;
    // the whole warp writes the chunk's decay tables; one lane issues a
    // forward chunk's C B^T once its tiles have landed.
    if (lane == 0) {
      prefetch_tmap(&map_x);
      prefetch_tmap(&map_b);
      prefetch_tmap(&map_c);
    }
    struct PUnit {
      long long b, e;
      int u, s, h, sigma, g, n, last_seg, tb, te;
      float A2;
    };
    auto draw = [&](PUnit& X) -> bool {
      int v = 0;
      if (lane == 0) v = atomicAdd(prm.ticket, 1);
      v = __shfl_sync(0xffffffffu, v, 0);
      if (v >= nunits) return false;
      X.u = v;
      X.s = upper_index(prm.uoff, nseq, v);
      const int rem = v - prm.uoff[X.s];
      X.sigma = rem / prm.H;
      X.h = rem % prm.H;
      X.g = (int)((long long)X.h * prm.G / prm.H);
      X.A2 = prm.A[X.h] * kLog2e;
      X.b = prm.si.begin(X.s);
      X.e = prm.si.end(X.s);
      const int nt = (int)((X.e - X.b + kQ - 1) / kQ);
      X.tb = X.sigma * prm.seg;
      X.te = min(nt, X.tb + prm.seg);
      X.last_seg = X.te == nt;
      X.n = X.te - X.tb;
      return true;
    };
    auto tile_of = [&](const PUnit& X, int k, long long& t0, int& kind, int& len) {
      kind = k < X.n ? kKindA : kKindB;
      const int t = kind == kKindA ? X.te - 1 - k : X.tb + (k - X.n);
      t0 = X.b + (long long)t * kQ;
      len = (int)min((long long)kQ, X.e - t0);
    };
    uint32_t it = 0;
    bool ok = true;
    PUnit U;
    int k = 0;
    bool have = plan_ok && draw(U);
    long long nt0 = 0;
    int nkind = 0, nlen = 0;
    __nv_bfloat16 dpre[4];
    auto load_dt = [&](const PUnit& X, long long t0, int len) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = 4 * lane + q;
        dpre[q] = j < len ? prm.dt[(t0 + j) * prm.H + X.h] : __float2bfloat16(0.f);
      }
    };
    if (have) {
      tile_of(U, 0, nt0, nkind, nlen);
      load_dt(U, nt0, nlen);
    }
    while (have) {
      const PUnit C = U;
      const long long t0 = nt0;
      const int kind = nkind, len = nlen;
      __nv_bfloat16 dcur[4];
      float dv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dcur[q] = dpre[q];
        dv[q] = __bfloat162float(dpre[q]);
      }
      if (++k >= 2 * U.n) {
        k = 0;
        have = draw(U);
      }
      if (have) {
        tile_of(U, k, nt0, nkind, nlen);
        load_dt(U, nt0, nlen);
      }
      const int cb = it & 1, xs = x_slot(it);
      bool good = it < kCB || wait_bar_warp(&bars[kCbEmpty0 + cb], cb_par(it - kCB), wns);
      if (good && it >= kXS) good = wait_bar_warp(&bars[kXEmpty0 + xs], x_par(it - kXS), wns);
      if (!good) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, *abort_v)) { ok = false; break; }
      uint64_t* fcb = &bars[kCbFull0 + cb];
      uint64_t* fx = &bars[kXFull0 + xs];
      if (lane == 0) {
        const int row = (int)t0;
        mbar_arrive_expect_tx(fx, kTile);
        tma_load_2d(sm.X(xs), &map_x, fx, C.h * kP, row);
        mbar_arrive_expect_tx(fcb, kind == kKindB ? 4 * kTile : 2 * kTile);
        tma_load_2d(sm.B(cb, 0), &map_b, fcb, C.g * kN, row);
        tma_load_2d(sm.B(cb, 1), &map_b, fcb, C.g * kN + 64, row);
        if (kind == kKindB) {
          tma_load_2d(sm.C(cb, 0), &map_c, fcb, C.g * kN, row);
          tma_load_2d(sm.C(cb, 1), &map_c, fcb, C.g * kN + 64, row);
        }
        // the next chunk's x into L2 behind this chunk's loads
        if (have) tma_prefetch_2d(&map_x, U.h * kP, (int)nt0);
        TileInfo* inf = sm.info(xs);
        inf->t0 = t0;
        inf->s = C.s;
        inf->h = C.h;
        inf->sigma = C.sigma;
        inf->unit = C.u;
        inf->len = len;
        inf->kind = kind;
        inf->cnt = C.n;
        inf->last_seg = C.last_seg;
      }
      // decay tables: lane l owns tokens 4l .. 4l+3
      float pre[4], run = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        run += dv[q] * C.A2;
        pre[q] = run;
      }
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float tv = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += tv;
      }
      const float excl = incl - run;
      float* c2t = sm.c2(xs);
      float* Et = sm.E(xs);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float cq2 = excl + pre[q];
        c2t[4 * lane + q] = cq2;
        Et[4 * lane + q] = 4 * lane + q < len ? fast_exp2(-cq2) * dv[q] : 0.f;
        sm.dt(xs)[4 * lane + q] = dcur[q];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(fx);
      ++it;
    }
    // sentinel: no more work (in the next x slot)
    const int xs = x_slot(it);
    if (ok && (it < kXS || wait_bar_warp(&bars[kXEmpty0 + xs], x_par(it - kXS), wns))) {
      if (lane == 0) {
        sm.info(xs)->kind = kKindEnd;
        mbar_arrive(&bars[kXFull0 + xs]);
        mbar_arrive(&bars[kXFull0 + xs]);
      }
    } else if (lane == 0) {
      if (ok) fail(SSD_ERR_TIMEOUT);
      // aborting: loads still in flight must land before the CTA may exit
      for (uint32_t q = (it >= kXS ? it - kXS : 0); q < it; ++q)
        (void)wait_bar(&bars[kXFull0 + x_slot(q)], x_par(q), wns);
      for (uint32_t q = (it >= kCB ? it - kCB : 0); q < it; ++q)
        (void)wait_bar(&bars[kCbFull0 + (q & 1)], cb_par(q), wns);
    }
  } else if (warp == kGWarp) {
    // ------------------------------------------------------------ C B^T issuer
    // Follows the chunks through the x slots (the tile info): each forward
    // chunk's C B^T once its C/B slot has landed and its S buffer is free;
    // it also gives the C/B slot its first release arrival (for a segment-
    // state chunk at once, for a forward chunk when C B^T has read it).
    uint32_t it = 0, gu = 0;
    bool issued = false;
    while (true) {
      const int cb = it & 1, xs = x_slot(it);
      bool good = wait_bar_warp(&bars[kXFull0 + xs], x_par(it), wns);
      if (!good) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        break;
      }
      const int kind = sm.info(xs)->kind;
      if (kind == kKindEnd || *abort_v) break;
      if (kind == kKindB) {
        good = wait_bar_warp(&bars[kCbFull0 + cb], cb_par(it), wns);
        if (good && gu >= 2) good = wait_bar_warp(&bars[kSFree0 + (gu & 1)], par2_of(gu - 2), wns);
        if (!good) {
          if (lane == 0) fail(SSD_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dC0 = sdesc_sw128(smem_u32(sm.C(cb, 0)), 16, 1024);
          const uint64_t dB0 = sdesc_sw128(smem_u32(sm.B(cb, 0)), 16, 1024);
          const uint32_t d = tmem + kColS + (gu & 1) * 128;
          // K steps of 32 bytes inside each 64-column half tile
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(d, dC0 + (kk >> 2) * kT16 + (kk & 3) * 2,
                     dB0 + (kk >> 2) * kT16 + (kk & 3) * 2, idG, kk > 0);
          mma_commit(&bars[kGFull0 + (gu & 1)]);
          mma_commit(&bars[kCbEmpty0 + cb]);
        }
        __syncwarp();
        issued = true;
        ++gu;
      } else if (lane == 0) {
        mbar_arrive(&bars[kCbEmpty0 + cb]);
      }
      ++it;
    }
    if (lane == 0) {
      // this warp's products must complete before tensor memory is freed
      if (issued) mma_commit(&bars[kMmaDone]);
      else mbar_arrive(&bars[kMmaDone]);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and bookkeeping are warp-uniform,
    // so descriptors live in uniform registers); one elected lane issues.
    // Descriptors are built once per buffer and advanced by constant
    // offsets (a descriptor's address field is bytes >> 4).
    const uint64_t dC0 = sdesc_sw128(smem_u32(sm.C(0, 0)), 16, 1024);       // K-major C
    const uint64_t dBt0 = sdesc_sw128(smem_u32(sm.B(0, 0)), kTile, 1024);   // MN-major B^T
    const uint64_t dW0 = sdesc_sw128(smem_u32(sm.W(0)), kTile, 1024);       // [w o X hi | lo]
    const uint64_t dX0 = sdesc_sw128(smem_u32(sm.X(0)), kTile, 1024);       // MN-major x
    const uint64_t dHt = sdesc_sw128(smem_u32(sm.Ht()), kTile, 1024);       // [H hi | lo]^T
    constexpr uint64_t kCB16 = kCBBytes >> 4;
    uint32_t it = 0, hu = 0, gu = 0, au = 0;
    uint32_t wa0 = 0, wa1 = 0;  // segment-state chunks that used C/B slot 0 / 1
    bool issued = false;
#define MMA_WAIT(bar, par)                      \
  if (!wait_bar_warp(&bars[bar], (par), wns)) { \
    if (lane == 0) fail(SSD_ERR_TIMEOUT);       \
    goto mma_done;                              \
  }
    while (true) {
      MMA_WAIT(kXFull0 + x_slot(it), x_par(it));
      if (sm.info(x_slot(it))->kind == kKindEnd || *abort_v) break;
      const int n = sm.info(x_slot(it))->cnt;
      // ---- segment-state pass: S_c = B^T [w o X hi | lo] per chunk
      for (int k = 0; k < n; ++k) {
        const int cb = it & 1, xs = x_slot(it);
        uint32_t& wa = cb ? wa1 : wa0;
        MMA_WAIT(kCbFull0 + cb, cb_par(it));
        MMA_WAIT(kWxFull0 + cb, par_of(wa));
        ++wa;
        if (au >= 2) { MMA_WAIT(kAccFree0 + (au & 1), par2_of(au - 2)); }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t d = tmem + kColAcc + (au & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(d, dBt0 + cb * kCB16 + kk * 128, dW0 + cb * kCB16 + kk * 128, idSt, kk > 0);
          mma_commit(&bars[kAccFull0 + (au & 1)]);
          mma_commit(&bars[kCbEmpty0 + cb]);
          mma_commit(&bars[kXEmpty0 + xs]);
        }
        __syncwarp();
        issued = true;
        ++au;
        ++it;
      }
      // ---- forward chunks: [C H_hi^T + S' X | C H_lo^T]
      for (int t = 0; t < n; ++t) {
        const int cb = it & 1, xs = x_slot(it);
        MMA_WAIT(kCbFull0 + cb, cb_par(it));
        MMA_WAIT(kHtFull, par_of(hu));
        if (au >= 2) { MMA_WAIT(kAccFree0 + (au & 1), par2_of(au - 2)); }
        tc_fence_after();
        const uint32_t d = tmem + kColAcc + (au & 1) * 128;
        if (elect_one()) {
          // C (K-major: K steps of 32 bytes inside each 64-column half tile)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(d, dC0 + cb * kCB16 + (kk >> 2) * kT16 + (kk & 3) * 2, dHt + kk * 128, idCH,
                     kk > 0);
          mma_commit(&bars[kHtFree]);
          mma_commit(&bars[kCbEmpty0 + cb]);
        }
        __syncwarp();
        MMA_WAIT(kXFull0 + xs, x_par(it));
        MMA_WAIT(kSFull0 + (gu & 1), par2_of(gu));
        tc_fence_after();
        if (elect_one()) {
          const uint32_t scol = tmem + kColS + (gu & 1) * 128;
          // S' from tensor memory: K block kk (columns j = 16 kk .. 16 kk + 15)
          // holds 8 columns of hi pairs, then 8 of lo pairs
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_tmem_a(d, scol + 16 * kk + 8 * part, dX0 + xs * kT16 + kk * 128, idSX, true);
          mma_commit(&bars[kAccFull0 + (au & 1)]);
          mma_commit(&bars[kSFree0 + (gu & 1)]);
          mma_commit(&bars[kXEmpty0 + xs]);
        }
        __syncwarp();
        issued = true;
        ++gu;
        ++hu;
        ++au;
        ++it;
      }
    }
  mma_done:
#undef MMA_WAIT
    // every product issued must complete before tensor memory is freed
    if (lane == 0) {
      if (issued) mma_commit(&bars[kMmaDone]);
      else mbar_arrive(&bars[kMmaDone]);
      if (!wait_bar(&bars[kMmaDone], 0, wns)) fail(SSD_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ math warps
    // Warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31 (a warp
    // may only touch its own lane quarter) and takes column quarter cq = w / 4.
    const int q = warp & 3;
    const int cq = warp >> 2;
    const int r = 32 * q + lane;  // tensor-memory lane: token row i / state row n
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t it = 0, hu = 0, gu = 0, au = 0, nsync = 0;
    // fp32 running state: pair k holds H[p][n = r] for p = 16 cq + 2k, 2k + 1
    f2 h2[8];
    // this thread's 16 values of a chunk state in the CTA's scratch: 64
    // contiguous bytes per thread (slot 0; slots are kPN floats apart)
    float* const stb = prm.stbuf + (long long)blockIdx.x * kStSlots * kPN + tid * 16;

    auto arrive = [&](int bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bar]);
    };

    // one 16-byte work item of w o X (items k = 0..1023: 8 values of row
    // j = k / 8), weight w_j = exp2(wl - c2_j) dt_j, written as bf16 hi and
    // lo tiles at `dst`
    auto wx_item = [&](int xs, int k, float wl, uint8_t* dst) {
      const int j = k >> 3, c = k & 7;
      const uint32_t off = sw128_offset(j, c);
      const uint4 xv = *reinterpret_cast<const uint4*>(sm.X(xs) + off);
      const float w = fast_exp2(wl - sm.c2(xs)[j]) * __bfloat162float(sm.dt(xs)[j]);
      const f2 ww{w, w};
      uint4 hi, lo;
      split2p(mul2(bf2(xv.x), ww), hi.x, lo.x);
      split2p(mul2(bf2(xv.y), ww), hi.y, lo.y);
      split2p(mul2(bf2(xv.z), ww), hi.z, lo.z);
      split2p(mul2(bf2(xv.w), ww), hi.w, lo.w);
      *reinterpret_cast<uint4*>(dst + off) = hi;
      *reinterpret_cast<uint4*>(dst + kTile + off) = lo;
    };

    // The mask S' of forward chunk number `pgu` (in S buffer pgu & 1), over
    // its C B^T in place: this warp's 32 x 32 block (rows 32 q.., columns
    // 32 cq..), in two 16-column halves, each rewritten as one K block: 8
    // columns of hi pairs followed by 8 of lo pairs.  Blocks above the
    // diagonal become zeros.
    auto build_mask = [&](uint32_t pgu, int xs, float c2r, float Dh) -> bool {
      const int gb = pgu & 1;
      if (!wait_bar_warp(&bars[kGFull0 + gb], par2_of(pgu), wns)) return false;
      tc_fence_after();
      const uint32_t scol = tmem + kColS + gb * 128 + lane_addr + 32 * cq;
      if (cq > q) {
        uint32_t z[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) z[m] = 0u;
        tmem_st16(scol, z);
        tmem_st16(scol + 16, z);
      } else {
        const bool diag = cq == q;
        const bool fast = __all_sync(0xffffffffu, c2r >= kDeep);
        const float mr = fmaxf(c2r, kDeep);
        const float Dr = Dh * fast_exp2(-mr);
        const float dr = c2r - mr;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int j0 = 32 * cq + 16 * half;
          float g[16];
          tmem_ld16(scol + 16 * half, g);
          tmem_ld_wait();
          tie16(g);
          f2 v[8];
          if (fast) {
            // every row's factor is exp(cum_i): S' = G E_j
            const float4* E4 = reinterpret_cast<const float4*>(sm.E(xs) + j0);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float4 e = E4[m];
              v[2 * m] = mul2(f2{g[4 * m], g[4 * m + 1]}, f2{e.x, e.y});
              v[2 * m + 1] = mul2(f2{g[4 * m + 2], g[4 * m + 3]}, f2{e.z, e.w});
            }
          } else {
            // some rows decayed below 2^-60: exp2(c2_i - m_i - c2_j) dt_j per entry
            const float4* c4 = reinterpret_cast<const float4*>(sm.c2(xs) + j0);
            const uint2* d2 = reinterpret_cast<const uint2*>(sm.dt(xs) + j0);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float4 cc = c4[m];
              const uint2 db = d2[m];
              const f2 e01 = mul2(f2{fast_exp2(dr - cc.x), fast_exp2(dr - cc.y)}, bf2(db.x));
              const f2 e23 = mul2(f2{fast_exp2(dr - cc.z), fast_exp2(dr - cc.w)}, bf2(db.y));
              v[2 * m] = mul2(f2{g[4 * m], g[4 * m + 1]}, e01);
              v[2 * m + 1] = mul2(f2{g[4 * m + 2], g[4 * m + 3]}, e23);
            }
          }
          if (diag) {
            // causal; the skip term rides on the diagonal
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) {
              const int c0 = 16 * half + 2 * pp, c1 = c0 + 1;
              v[pp].x = c0 < lane ? v[pp].x : (c0 == lane ? v[pp].x + Dr : 0.f);
              v[pp].y = c1 < lane ? v[pp].y : (c1 == lane ? v[pp].y + Dr : 0.f);
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int pp = 0; pp < 8; ++pp) split2p(v[pp], pk[pp], pk[8 + pp]);
          tmem_st16(scol + 16 * half, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      arrive(kSFull0 + gb);
      return true;
    };

    // H^T (hi, lo) as the B operand of C H^T: row n = r, columns p = 16 cq..
    auto put_ht = [&]() -> bool {
      if (hu >= 1 && !wait_bar_warp(&bars[kHtFree], par_of(hu - 1), wns)) return false;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint4 h4, l4;
        split2p(h2[4 * c + 0], h4.x, l4.x);
        split2p(h2[4 * c + 1], h4.y, l4.y);
        split2p(h2[4 * c + 2], h4.z, l4.z);
        split2p(h2[4 * c + 3], h4.w, l4.w);
        const uint32_t off = sw128_offset(r, 2 * cq + c);
        *reinterpret_cast<uint4*>(sm.Ht() + off) = h4;
        *reinterpret_cast<uint4*>(sm.Ht() + kTile + off) = l4;
      }
      fence_proxy_async_smem();
      arrive(kHtFull);
      ++hu;
      return true;
    };

    // This thread's 16 columns of accumulator use `au` (lane r, columns
    // 16 cq.. of both 64-column halves, summed), 8 at a time: `use(c0, v)`
    // receives columns 16 cq + c0 .. + 7.  Then the buffer goes back.
    auto with_acc = [&](auto&& use) -> bool {
      const int ab = au & 1;
      if (!wait_bar_warp(&bars[kAccFull0 + ab], par2_of(au), wns)) return false;
      tc_fence_after();
      const uint32_t base = tmem + kColAcc + ab * 128 + lane_addr + 16 * cq;
#pragma unroll
      for (int c0 = 0; c0 < 16; c0 += 8) {
        float a[8], b[8];
        tmem_ld8(base + c0, a);
        tmem_ld8(base + 64 + c0, b);
        tmem_ld_wait();
        tie8(a);
        tie8(b);
        if (c0 == 8) {
          tc_fence_before();
          arrive(kAccFree0 + ab);
          ++au;
        }
        f2 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = add2(f2{a[2 * k], a[2 * k + 1]}, f2{b[2 * k], b[2 * k + 1]});
        use(c0, v);
      }
      return true;
    };

    // y = f (S' X + C H^T) of the forward chunk whose accumulator is next
    auto epilogue = [&](float f, long long t0, int len, int h) -> bool {
      float* yp = prm.y + ((t0 + r) * prm.H + h) * kP + 16 * cq;
      const bool row_ok = r < len;
      return with_acc([&](int c0, f2 (&v)[4]) {
        float o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const f2 t = mul2(v[k], f2{f, f});
          o[2 * k] = t.x;
          o[2 * k + 1] = t.y;
        }
        if (row_ok) {
          if (prm.y_v8) {
            st_global_cs_v8(yp + c0, o);
          } else {
            __stcs(reinterpret_cast<float4*>(yp + c0), make_float4(o[0], o[1], o[2], o[3]));
            __stcs(reinterpret_cast<float4*>(yp + c0) + 1, make_float4(o[4], o[5], o[6], o[7]));
          }
        }
      });
    };

    // the chunk state in scratch slot `slot` has been consumed: each warp
    // drops its 2 KB (16 lines) from L2 unwritten
    auto discard_slot = [&](int slot) {
      __syncwarp();
      if (lane < 16) discard_l2_line(stb - tid * 16 + (long long)slot * kPN + warp * 512 + lane * 32);
    };
    // this thread's 16 values of the chunk state in scratch slot `slot`
    auto load_slot = [&](int slot, f2 (&sv)[8]) {
      const float4* src = reinterpret_cast<const float4*>(stb + (long long)slot * kPN);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 t = __ldcg(src + c);
        sv[2 * c] = f2{t.x, t.y};
        sv[2 * c + 1] = f2{t.z, t.w};
      }
    };

#define MATH_TRY(expr)     \
  if (!(expr)) {           \
    fail(SSD_ERR_TIMEOUT); \
    goto math_done;        \
  }
    while (true) {
      MATH_TRY(wait_bar_warp(&bars[kXFull0 + x_slot(it)], x_par(it), wns));
      if (sm.info(x_slot(it))->kind == kKindEnd || __any_sync(0xffffffffu, *abort_v)) break;
      const TileInfo u0 = *sm.info(x_slot(it));
      const int h = u0.h, n = u0.cnt;
      const float Dh = prm.D ? prm.D[h] : 0.f;
      // the initial state of a sequence's first segment: into L2 now, read at
      // the hand-off
      const float* ini = (u0.sigma == 0 && prm.init)
                             ? prm.init + ((long long)u0.s * prm.H + h) * kPN : nullptr;
      if (ini && lane < 16) prefetch_l2(ini + (16 * cq + lane) * kN + 32 * q);

      // -------- segment-state pass: each chunk's state S_c (chunk-local
      // weights w_j = exp(cum_last - cum_j) dt_j), chunks walked backwards,
      // kept in scratch slot (its index in the segment) and folded into
      // H_loc = sum_c exp(sum of the later chunks' dt A) S_c.  The w o X
      // tiles go into the C half of the chunk's C/B slot.
      f2 hloc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) hloc[k] = f2{0.f, 0.f};
      float later = 0.f;  // log2-decay of the chunks already folded (later in time)
      auto fold = [&](int kk, float c2l_kk) -> bool {
        const float wl = fast_exp2(later);
        float4* dst = reinterpret_cast<float4*>(stb + (long long)(n - 1 - kk) * kPN);
        const bool ok = with_acc([&](int c0, f2 (&v)[4]) {
          __stcg(dst + c0 / 4, make_float4(v[0].x, v[0].y, v[1].x, v[1].y));
          __stcg(dst + c0 / 4 + 1, make_float4(v[2].x, v[2].y, v[3].x, v[3].y));
#pragma unroll
          for (int k = 0; k < 4; ++k) hloc[c0 / 2 + k] = fma2(f2{wl, wl}, v[k], hloc[c0 / 2 + k]);
        });
        later += c2l_kk;
        return ok;
      };
      float c2l_prev = 0.f;
      for (int k = 0; k < n; ++k) {
        const int cb = it & 1, xs = x_slot(it);
        if (k > 0) MATH_TRY(wait_bar_warp(&bars[kXFull0 + xs], x_par(it), wns));
        // the slot's B tile has landed, and with it the slot is free of its
        // previous chunk: w o X may be written into its C half
        MATH_TRY(wait_bar_warp(&bars[kCbFull0 + cb], cb_par(it), wns));
        const float c2l = sm.c2(xs)[kQ - 1];
        wx_item(xs, tid, c2l, sm.W(cb));
        wx_item(xs, tid + 512, c2l, sm.W(cb));
        fence_proxy_async_smem();
        arrive(kWxFull0 + cb);
        arrive(kXEmpty0 + xs);
        // the previous chunk's product, read while this one's is computed
        if (k > 0) MATH_TRY(fold(k - 1, c2l_prev));
        c2l_prev = c2l;
        ++it;
      }
      MATH_TRY(fold(n - 1, c2l_prev));

      // -------- the first forward chunk's mask does not need the incoming
      // state: build it while the predecessor may still be publishing
      const int xs0 = x_slot(it);
      MATH_TRY(wait_bar_warp(&bars[kXFull0 + xs0], x_par(it), wns));
      MATH_TRY(build_mask(gu, xs0, sm.c2(xs0)[r], Dh));
      ++gu;

      // -------- segment hand-off
      if (u0.sigma == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          h2[k] = ini ? f2{__ldg(ini + (16 * cq + 2 * k) * kN + r), __ldg(ini + (16 * cq + 2 * k + 1) * kN + r)}
                      : f2{0.f, 0.f};
      } else {
        const int pred = u0.unit - prm.H;  // same sequence and head, previous segment
        if (tid == 0) {
          const unsigned long long t0 = gtime();
#pragma unroll 1
          for (uint32_t m = 1; ld_acquire(prm.flags + pred) == 0; ++m) {
            __nanosleep(200);
            if ((m & 15u) == 0 && gtime() - t0 > wns) {
              fail(SSD_ERR_TIMEOUT);
              break;
            }
          }
        }
        MATH_TRY(math_sync(&bars[kSync], par_of(nsync), wns));
        ++nsync;
        if (__any_sync(0xffffffffu, *abort_v)) goto math_done;
        const float* src = prm.slots + (long long)pred * kPN;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          h2[k] = f2{__ldcg(src + (16 * cq + 2 * k) * kN + r), __ldcg(src + (16 * cq + 2 * k + 1) * kN + r)};
      }
      if (!u0.last_seg) {
        const float aseg = fast_exp2(later);
        float* dst = prm.slots + (long long)u0.unit * kPN;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const f2 e = fma2(f2{aseg, aseg}, h2[k], hloc[k]);
          __stcg(dst + (16 * cq + 2 * k) * kN + r, e.x);
          __stcg(dst + (16 * cq + 2 * k + 1) * kN + r, e.y);
        }
        MATH_TRY(math_sync(&bars[kSync], par_of(nsync), wns));
        ++nsync;
        if (tid == 0 && u0.unit != prm.hold_unit) {
          __threadfence();
          st_release(prm.flags + u0.unit, 1);
        }
      }
      // the state entering the segment feeds the first chunk's C H^T
      MATH_TRY(put_ht());

      // -------- forward chunks.  Iteration t: the state after chunk t (H^T
      // for chunk t + 1's C H^T), the mask of chunk t + 1, chunk t's y.
      f2 sv[8];
      load_slot(0, sv);
      for (int t = 0; t < n; ++t) {
        const int xs = x_slot(it);
        // this chunk's values (its x slot is full: its mask was built)
        const float a = fast_exp2(sm.c2(xs)[kQ - 1]);
        const float f = fast_exp2(fmaxf(sm.c2(xs)[r], kDeep));
        const long long t0 = sm.info(xs)->t0;
        const int len = sm.info(xs)->len;
        arrive(kXEmpty0 + xs);
#pragma unroll
        for (int k = 0; k < 8; ++k) h2[k] = fma2(f2{a, a}, h2[k], sv[k]);
        discard_slot(t);
        if (t + 1 < n) {
          load_slot(t + 1, sv);  // in flight during the mask and the epilogue
          MATH_TRY(put_ht());
          const int xn = x_slot(it + 1);
          MATH_TRY(wait_bar_warp(&bars[kXFull0 + xn], x_par(it + 1), wns));
          MATH_TRY(build_mask(gu, xn, sm.c2(xn)[r], Dh));
          ++gu;
        } else if (u0.last_seg && prm.final_states) {
          // the sequence's final state
          float* fin = prm.final_states + ((long long)u0.s * prm.H + h) * kPN;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            fin[(16 * cq + 2 * k) * kN + r] = h2[k].x;
            fin[(16 * cq + 2 * k + 1) * kN + r] = h2[k].y;
          }
        }
        MATH_TRY(epilogue(f, t0, len, h));
        ++it;
      }
    }
  math_done:;
#undef MATH_TRY
  }

#undef fail
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}

struct WsLayout {
  size_t uoff, ticket, flags, slots, stbuf, total;
};

WsLayout ws_layout(const FwdArgs& a) {
  WsLayout L;
  const long long mu = tc_max_units(a);
  L.uoff = 0;
  L.ticket = L.uoff + plan_bytes(a.nseq);
  L.flags = L.ticket + 256;
  L.slots = L.flags + align256(sizeof(int) * (size_t)mu);
  L.stbuf = L.slots + align256(sizeof(float) * (size_t)mu * kPN);
  L.total = L.stbuf + align256(sizeof(float) * (size_t)tc_sm_count() * kStSlots * kPN);
  return L;
}

}  // namespace

bool tc2_supported(const FwdArgs& a) {
  return a.dtype == SSD_DT_BF16 && a.P == kP && a.N == kN && !a.dt_softplus && !a.z &&
         !a.y_bf16;
}

size_t tc2_workspace_bytes(const FwdArgs& a) { return ws_layout(a).total; }

ssd_status_t tc2_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit) {
  const WsLayout L = ws_layout(a);
  char* ws = static_cast<char*>(a.ws);
  int32_t* uoff = reinterpret_cast<int32_t*>(ws + L.uoff);
  int* ticket = reinterpret_cast<int*>(ws + L.ticket);
  int* flags = reinterpret_cast<int*>(ws + L.flags);
  float* slots = reinterpret_cast<float*>(ws + L.slots);
  float* stbuf = reinterpret_cast<float*>(ws + L.stbuf);
  const long long ntok = (long long)a.batch * a.seqlen;
  const long long mu = tc_max_units(a);
  const int seg = tc_choose_seg(a);
  // everything the host prepares comes before the first launch, so the two
  // kernels reach the GPU back to back
  CUtensorMap mx, mb, mc;
  const bool work = ntok > 0 && mu > 0;
  if (work && (!tc_make_map_bf16(&mx, a.x, ntok, (long long)a.H * kP) ||
               !tc_make_map_bf16(&mb, a.B, ntok, (long long)a.G * kN) ||
               !tc_make_map_bf16(&mc, a.C, ntok, (long long)a.G * kN)))
    return SSD_ERR_CUDA;
  Params p;
  p.dt = static_cast<const __nv_bfloat16*>(a.dt);
  p.A = a.A;
  p.D = a.D;
  p.init = a.init;
  p.y = a.y;
  p.final_states = a.final_states;
  p.si = SeqInfo{a.cu, a.seqlen, a.nseq};
  p.uoff = uoff;
  p.ticket = ticket;
  p.flags = flags;
  p.slots = slots;
  p.stbuf = stbuf;
  p.status = a.dev_status;
  p.H = a.H;
  p.G = a.G;
  p.seg = seg;
  p.y_v8 = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
  p.wait_ns = wait_ns;
  p.hold_unit = hold_unit;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(ssd_fwd2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;
  if (tc_launch_plan(a, seg, uoff, ticket, flags, mu) != cudaSuccess) return SSD_ERR_CUDA;
  if (!work) return SSD_OK;
  const int grid = (int)(mu < tc_sm_count() ? mu : tc_sm_count());
  // Programmatic dependent launch: the forward kernel may start while the
  // plan kernel runs; it waits for the plan's results (griddepcontrol.wait)
  // after its own set-up (barriers, tensor memory, tensor-map prefetch).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, ssd_fwd2_kernel, mx, mb, mc, p) != cudaSuccess) return SSD_ERR_CUDA;
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
