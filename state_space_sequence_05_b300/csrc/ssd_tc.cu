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
// D_h x is folded into Y_diag: D_h sits on the diagonal of S.
//
// Precision: x, B and C arrive in bf16 and are used as they are.  The three
// operands the kernel derives (S, w o X and H) are fp32 values; each is
// written as a pair of bf16 numbers, hi = v truncated to bf16 and lo = (v -
// hi) truncated to bf16 (|v - hi - lo| < 2^-14 |v|), and both halves are
// multiplied into the same fp32 accumulator.  (A single bf16 rounding of any
// one of these operands costs about 1-5e-2 of RMS(y) in max error.)
//
// The chunk length is fixed at 128 = the tcgen05 tile height M.  Any chunk
// size gives the same function up to rounding (the decomposition is an
// exact reordering of the recurrence), so every chunk_size the API accepts
// runs with 128-token blocks here.
//
// Work partition.  Each sequence is cut into segments of 4-12 chunks; a
// work unit is one (sequence, segment, head), handed out in that order by a
// global ticket, so a unit's predecessor (same sequence and head, previous
// segment) was always taken earlier by a running CTA.  A unit
//   1. computes each chunk's state S_c = B^T (w o X) on the tensor cores,
//      walking the chunks backwards, keeps them in a per-CTA scratch (L2-
//      resident; every thread reloads only what it stored) and folds them
//      into the segment-local state H_loc, the decayed sum of its chunk
//      states from a zero state;
//   2. takes the state entering the segment, H_in, from the initial state
//      (first segment) or from its predecessor's published end state, and
//      publishes its own end state exp(sum of the segment's dt A) H_in +
//      H_loc with a release flag: the inter-chunk recurrence carried across
//      CTAs at segment granularity, i.e. the composition of affine maps
//      (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2) ("Mamba ... review",
//      feghi.github.io, sec. 4);
//   3. runs the forward over its chunks starting from H_in, with
//      H_c = exp(cum_last) H_{c-1} + S_c from the kept chunk states.
// The running state never leaves the SM between the chunks of a segment.
//
// Roles (one persistent CTA per SM, 576 threads):
//   warp 16    TMA producer: C, B, x tiles (128B swizzle) into a 2-stage ring,
//              and the chunk's cumulative decay table.
//   warp 17    MMA issuer (one thread): C B^T, B^T (w o X), C H^T and S X
//              (S read from tensor memory); issues the next chunk's C B^T
//              ahead of the current chunk's products.
//   warps 0-15 CUDA-core math (TMEM lane quarter w % 4, column quarter
//              w / 4): decay mask (built for chunk c+1 while the tensor core
//              works on chunk c), w o X, fp32 state in registers, epilogue,
//              segment hand-off.
// Every wait is bounded in time; on expiry the kernel records
// SSD_ERR_TIMEOUT and unwinds.
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

constexpr int kQ = 128;  // chunk tokens = MMA M
constexpr int kP = 64;   // headdim
constexpr int kN = 128;  // dstate
constexpr int kPN = kP * kN;
constexpr int kStages = 2;
constexpr int kMathWarps = 16;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;

constexpr uint32_t kTile = 16384;                   // one 128 x 64 bf16 tile
constexpr uint32_t kStageBytes = 5 * kTile;         // C0 C1 B0 B1 X
constexpr uint32_t kStageBytesA = 3 * kTile;        // B0 B1 X (segment-state pass)
constexpr uint32_t kOffXw = kStages * kStageBytes;  // w o X as bf16 hi, lo (2 x 16 KB)
constexpr uint32_t kOffHt = kOffXw + 2 * kTile;     // H^T as bf16 hi, lo (2 x 16 KB)
// per stage: c2 fp32[128], E fp32[128], dt bf16[128]
constexpr uint32_t kOffTabs = kOffHt + 2 * kTile;
constexpr uint32_t kTabBytes = 128 * 4 + 128 * 4 + 128 * 2;  // c2, E, dt (bf16)
constexpr uint32_t kOffInfo = kOffTabs + kStages * kTabBytes;
constexpr uint32_t kOffBars = kOffInfo + 2 * 64;
// (barriers, then the TMEM base address and the abort flag)
constexpr uint32_t kBarBytes = 32 * 8;
constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 16;

// TMEM columns (fp32 accumulators, 128 lanes).
constexpr uint32_t kColCB = 0;     // 2 x 128: C B^T, overwritten in place by S (hi/lo pairs)
constexpr uint32_t kColYD = 256;   // 2 x 64: S X, double-buffered by forward chunk
constexpr uint32_t kColYO = 384;   // 128: C H_hi^T | C H_lo^T
// The segment-state pass puts each chunk's state product B^T [w o X hi |
// w o X lo] (lane n, columns p of the hi half, then of the lo half) in the
// columns of the two S buffers, alternating: S is not live during that pass.
constexpr uint32_t kColSA = 0;
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Chunks per unit, at most (segment lengths: see tc_choose_seg).
constexpr int kStSlots = kTcSegMax > kTcSegVarlen ? kTcSegMax : kTcSegVarlen;

enum : int { kKindA = 0, kKindB = 1, kKindEnd = 2 };

struct TileInfo {
  long long t0;  // first token of the chunk
  int s, h, sigma, unit;
  int len;       // valid rows (1..128)
  int kind;      // kKindA (segment-state pass), kKindB (forward), kKindEnd
  int idx, cnt;  // position of this chunk among the unit's chunks of its kind
  int nA;        // chunks in the unit's segment-state pass (0 = none)
  int last_seg;  // the unit is its sequence's last segment
  int ez;        // the E table is finite: |cum_last| log2(e) < 120
  int pad;
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

// Fused epilogue options (ssd_fwd_epilogue_t), read by the epilogue kernel
// variant only.
struct EpiParams {
  const float* dt_bias;         // [H] or null
  const __nv_bfloat16* z;       // [tokens, H * kP] or null: y *= silu(z)
  int dt_softplus;              // dt = softplus(dt + dt_bias[h]) in the tables
  int y_bf16;                   // y stored as bf16 (round to nearest even)
};

struct Smem {
  uint8_t* base;
  __device__ uint8_t* stage(int s) const { return base + s * kStageBytes; }
  __device__ uint8_t* C(int s, int half) const { return stage(s) + half * kTile; }
  __device__ uint8_t* B(int s, int half) const { return stage(s) + (2 + half) * kTile; }
  __device__ uint8_t* X(int s) const { return stage(s) + 4 * kTile; }
  __device__ uint8_t* Xw(int part) const { return base + kOffXw + part * kTile; }
  __device__ uint8_t* Ht(int part) const { return base + kOffHt + part * kTile; }
  // cumulative log2-decay of the chunk in stage s: c2[j] = sum_{k<=j} dt_k A log2(e)
  __device__ float* c2(int s) const {
    return reinterpret_cast<float*>(base + kOffTabs + s * kTabBytes);
  }
  // E[j] = exp(-cum_j) dt_j of the chunk in stage s (0 beyond the valid
  // rows).  In the fused-epilogue variant, whose dt is an fp32 softplus, the
  // slot holds E only when the tile info's `ez` is set (the chunk's decay
  // range keeps E finite) and dt_j itself otherwise; the bf16 dt table below
  // is then unused.
  __device__ float* E(int s) const {
    return reinterpret_cast<float*>(base + kOffTabs + s * kTabBytes + 512);
  }
  // dt of the chunk in stage s (0 beyond the valid rows)
  __device__ __nv_bfloat16* dt(int s) const {
    return reinterpret_cast<__nv_bfloat16*>(base + kOffTabs + s * kTabBytes + 1024);
  }
  __device__ TileInfo* info(int s) const {
    return reinterpret_cast<TileInfo*>(base + kOffInfo) + s;
  }
};

// barrier indices
enum {
  kFull0 = 0, kFull1, kEmpty0, kEmpty1,      // TMA stage ring
  kCbFull0, kCbFull1, kCbEmpty0, kCbEmpty1,  // C B^T / S buffers in TMEM
  kSFull0, kSFull1,                          // S written (math -> MMA), per S buffer
  kXwFull, kXwEmpty,                         // w o X buffer
  kXwFull1, kXwEmpty1,                       // pass A's second w o X buffer (the H^T tiles)
  kHFull, kHEmpty,                           // H^T buffer
  kAccFull,                                  // Y_diag, Y_off, chunk state ready
  kYoFree, kYdFree0, kYdFree1,               // each accumulator read (math -> MMA)
  kSaFull0, kSaFull1, kSaFree0, kSaFree1,    // segment-state chunk products in TMEM
  kYRead,                                    // staged y tiles read by their TMA stores
  kSyncHand,                                 // math-warp rendezvous
  kMmaDone,
  kNumBars
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

// kEpi: the fused-epilogue variant (dt = softplus(dt + dt_bias), y *=
// silu(z), bf16 y); it stores y directly instead of through the TMA staging
// tiles.  The plain variant carries none of that code.
template <bool kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_fwd_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_c,
                      const __grid_constant__ CUtensorMap map_y,
                      const __grid_constant__ CUtensorMap map_z, Params prm, EpiParams ep) {
  // All shared memory is dynamic: the tiles need 1024-byte alignment and
  // there is no room for a padding slack, so the base must come aligned.
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

  if (tid == 0) {
    mbar_init(&bars[kFull0], 2);  // expect-tx arrival + decay tables written
    mbar_init(&bars[kFull1], 2);
    mbar_init(&bars[kEmpty0], 1 + kMathWarps);
    mbar_init(&bars[kEmpty1], 1 + kMathWarps);
    mbar_init(&bars[kCbFull0], 1);
    mbar_init(&bars[kCbFull1], 1);
    mbar_init(&bars[kCbEmpty0], 1);
    mbar_init(&bars[kCbEmpty1], 1);
    mbar_init(&bars[kSFull0], kMathWarps);
    mbar_init(&bars[kSFull1], kMathWarps);
    mbar_init(&bars[kXwFull], kMathWarps);
    mbar_init(&bars[kXwEmpty], 1);
    mbar_init(&bars[kXwFull1], kMathWarps);
    mbar_init(&bars[kXwEmpty1], 1);
    mbar_init(&bars[kHFull], kMathWarps);
    mbar_init(&bars[kHEmpty], 1);
    mbar_init(&bars[kAccFull], 1);
    mbar_init(&bars[kYoFree], kMathWarps);
    mbar_init(&bars[kYdFree0], kMathWarps);
    mbar_init(&bars[kYdFree1], kMathWarps);
    mbar_init(&bars[kSaFull0], 1);
    mbar_init(&bars[kSaFull1], 1);
    mbar_init(&bars[kSaFree0], kMathWarps);
    mbar_init(&bars[kSaFree1], kMathWarps);
    mbar_init(&bars[kSyncHand], kMathWarps);
    mbar_init(&bars[kMmaDone], 1);
    mbar_init(&bars[kYRead], kMathWarps);
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Walks the ring one chunk at a time: a work unit (ticket), then its
    // segment-state chunks (backwards), then its forward chunks.  Lane 0
    // issues the TMA loads; the whole warp writes the chunk's decay tables.
    // The dt values of the next chunk are loaded one chunk ahead so their
    // latency overlaps the current chunk's hand-over.
    if (lane == 0) {
      prefetch_tmap(&map_x);
      prefetch_tmap(&map_b);
      prefetch_tmap(&map_c);
      prefetch_tmap(&map_y);
    }
    struct PUnit {
      long long b, e;
      int u, s, h, sigma, g, nA, nB, last_seg, tb, te;
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
      X.nA = X.te - X.tb;  // every unit keeps its chunk states (pass A)
      X.nB = X.te - X.tb;
      return true;
    };
    // first token, kind and valid rows of chunk k of unit X
    auto tile_of = [&](const PUnit& X, int k, long long& t0, int& kind, int& len) {
      kind = k < X.nA ? kKindA : kKindB;
      const int t = kind == kKindA ? X.te - 1 - k : X.tb + (k - X.nA);
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
      const int ck = k;
      const long long t0 = nt0;
      const int kind = nkind, len = nlen;
      float dv[4];
      __nv_bfloat16 dpre_cur[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dpre_cur[q] = dpre[q];
        dv[q] = __bfloat162float(dpre[q]);
      }
      if constexpr (kEpi) if (ep.dt_softplus) {
        // dt = softplus(dt + dt_bias[h]) on the valid rows (padding rows stay
        // 0): softplus(v) = max(v, 0) + log(1 + e), e = exp(-|v|) in (0, 1];
        // log(1 + e) = ln 2 * log2(1 + e), or e itself once e < 2^-12 (the
        // next term, e^2 / 2, is below 2^-13 e)
        const float bias = ep.dt_bias ? ep.dt_bias[C.h] : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float v = dv[q] + bias;
          const float e = fast_exp2(-fabsf(v) * kLog2e);
          const float l1p = e < 0x1p-12f ? e : kLn2 * fast_log2(1.f + e);
          dv[q] = 4 * lane + q < len ? fmaxf(v, 0.f) + l1p : 0.f;
        }
      }
      // advance, and start the next chunk's dt loads
      if (++k >= U.nA + U.nB) {
        k = 0;
        have = draw(U);
      }
      if (have) {
        tile_of(U, k, nt0, nkind, nlen);
        load_dt(U, nt0, nlen);
      }
      // hand this chunk over through stage it & 1
      const int st = it & 1;
      if (it >= 2 && !wait_bar_warp(&bars[kEmpty0 + st], ((it >> 1) - 1) & 1, prm.wait_ns)) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, *abort_v)) { ok = false; break; }
      uint64_t* fb = &bars[kFull0 + st];
      if (lane == 0) {
        // the loads first (x, from DRAM, the slowest), the tile info after:
        // the consumers read it only once this warp's table arrival lands
        const int row = (int)t0;
        mbar_arrive_expect_tx(fb, kind == kKindB ? kStageBytes : kStageBytesA);
        tma_load_2d(sm.X(st), &map_x, fb, C.h * kP, row);
        tma_load_2d(sm.B(st, 0), &map_b, fb, C.g * kN, row);
        tma_load_2d(sm.B(st, 1), &map_b, fb, C.g * kN + 64, row);
        if (kind == kKindB) {
          tma_load_2d(sm.C(st, 0), &map_c, fb, C.g * kN, row);
          tma_load_2d(sm.C(st, 1), &map_c, fb, C.g * kN + 64, row);
        }
        // the next chunk's x into L2, queued behind this chunk's loads (its
        // C and B tiles are shared by every head and are usually there
        // already)
        if (have) tma_prefetch_2d(&map_x, U.h * kP, (int)nt0);
        // the gate's z tile of a forward chunk, into L2 long before its epilogue
        if constexpr (kEpi)
          if (ep.z && kind == kKindB) tma_prefetch_2d(&map_z, C.h * kP, row);
        TileInfo* inf = sm.info(st);
        inf->t0 = t0;
        inf->s = C.s;
        inf->h = C.h;
        inf->sigma = C.sigma;
        inf->unit = C.u;
        inf->len = len;
        inf->kind = kind;
        inf->idx = kind == kKindA ? ck : ck - C.nA;
        inf->cnt = kind == kKindA ? C.nA : C.nB;
        inf->nA = C.nA;
        inf->last_seg = C.last_seg;
      }
      // decay table: lane l owns tokens 4l .. 4l+3
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
      float* c2t = sm.c2(st);
      float* Et = sm.E(st);
      // E[j] = exp(-cum_j) dt_j lets the mask and w o X use one table for
      // every column: exp(cum_i - cum_j) dt_j = exp(cum_i) E[j].  Valid
      // while the chunk's whole decay keeps both factors inside fp32
      const float tot = __shfl_sync(0xffffffffu, incl, 31);
      const bool ez = fabsf(tot) < 120.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float cq2 = excl + pre[q];
        c2t[4 * lane + q] = cq2;
        if constexpr (kEpi) {
          Et[4 * lane + q] = ez ? fast_exp2(-cq2) * dv[q] : dv[q];
        } else {
          Et[4 * lane + q] = fast_exp2(-cq2) * dv[q];
          sm.dt(st)[4 * lane + q] = dpre_cur[q];
        }
      }
      if (lane == 0) sm.info(st)->ez = ez;
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);
      ++it;
    }
    // sentinel: no more work
    const int st = it & 1;
    if (ok && (it < 2 || wait_bar_warp(&bars[kEmpty0 + st], ((it >> 1) - 1) & 1, prm.wait_ns))) {
      if (lane == 0) {
        sm.info(st)->kind = kKindEnd;
        mbar_arrive(&bars[kFull0 + st]);
        mbar_arrive(&bars[kFull0 + st]);
      }
    } else if (lane == 0) {
      if (ok) fail(SSD_ERR_TIMEOUT);
      // aborting: loads still in flight must land before the CTA may exit
      for (uint32_t q = (it >= 2 ? it - 2 : 0); q < it; ++q)
        (void)wait_bar(&bars[kFull0 + (q & 1)], (q >> 1) & 1, prm.wait_ns);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idCB = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idSA = idesc_bf16(128, 128, true, true);
      constexpr uint32_t idYO = idesc_bf16(128, 128, false, true);
      constexpr uint32_t idYD = idesc_bf16(128, 64, false, true);
      uint32_t it = 0, bt = 0, xu = 0, xu1 = 0, sa = 0;
      bool issued = false;
#define MMA_WAIT(bar, par)            \
  if (!wait_bar(&bars[bar], (par), prm.wait_ns)) { \
    fail(SSD_ERR_TIMEOUT);            \
    break;                            \
  }
      // C B^T of ring chunk `rit`, forward-chunk number `rbt`
      auto issue_cb = [&](uint32_t rit, uint32_t rbt) {
        const int st = rit & 1;
        const uint32_t cbcol = tmem + kColCB + (rbt & 1) * 128;
        const uint32_t aC0 = smem_u32(sm.C(st, 0)), aC1 = smem_u32(sm.C(st, 1));
        const uint32_t aB0 = smem_u32(sm.B(st, 0)), aB1 = smem_u32(sm.B(st, 1));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = (k & 3) * 32;
          mma_bf16(cbcol, sdesc_sw128((k < 4 ? aC0 : aC1) + kb, 16, 1024),
                   sdesc_sw128((k < 4 ? aB0 : aB1) + kb, 16, 1024), idCB, k > 0);
        }
        mma_commit(&bars[kCbFull0 + (rbt & 1)]);
      };
      while (true) {
        const int st = it & 1;
        MMA_WAIT(kFull0 + st, (it >> 1) & 1);
        const TileInfo inf = *sm.info(st);
        if (inf.kind == kKindEnd || *abort_v) break;
        tc_fence_after();
        const uint32_t aB0 = smem_u32(sm.B(st, 0));
        if (inf.kind == kKindA) {
          // segment-state pass: this chunk's state B^T [w o X hi | w o X lo],
          // one N = 128 product per K step, into the S columns (alternating
          // between the two S buffers); the math warps sum the halves and
          // keep the result.  The chunks also alternate between the w o X
          // tiles and the H^T tiles (H^T is not needed before the hand-off),
          // so one chunk's w o X is written while the tensor core reads the
          // previous one.
          if (inf.idx == 0) {
            // the previous unit's last S X products read the S columns
            if (bt >= 1) { MMA_WAIT(kCbEmpty0 + ((bt - 1) & 1), ((bt - 1) >> 1) & 1); }
            if (bt >= 2) { MMA_WAIT(kCbEmpty0 + ((bt - 2) & 1), ((bt - 2) >> 1) & 1); }
          }
          const int xb = inf.idx & 1;
          if (xb == 0) {
            MMA_WAIT(kXwFull, xu & 1);
          } else {
            MMA_WAIT(kXwFull1, xu1 & 1);
          }
          if (sa >= 2) { MMA_WAIT(kSaFree0 + (sa & 1), ((sa >> 1) - 1) & 1); }
          tc_fence_after();
          {
            const uint32_t aXw = smem_u32(xb == 0 ? sm.Xw(0) : sm.Ht(0));
            const uint32_t dcol = tmem + kColSA + (sa & 1) * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_bf16(dcol, sdesc_sw128(aB0 + k * 2048, kTile, 1024),
                       sdesc_sw128(aXw + k * 2048, kTile, 1024), idSA, k > 0);
          }
          issued = true;
          mma_commit(&bars[xb == 0 ? kXwEmpty : kXwEmpty1]);
          mma_commit(&bars[kEmpty0 + st]);
          mma_commit(&bars[kSaFull0 + (sa & 1)]);
          if (xb == 0) ++xu; else ++xu1;
          ++sa;
          ++it;
          continue;
        }
        // forward chunk: C B^T of this chunk if not issued ahead, then --
        // in whatever order their inputs become ready -- the next chunk's
        // C B^T (so the math warps can build its mask early), C H^T and S X.
        // The chunk state needs no product here: the segment-state pass
        // kept it.  Nothing waits behind an input that is late.
        if (inf.idx == 0) {
          if (bt >= 2) { MMA_WAIT(kCbEmpty0 + (bt & 1), ((bt >> 1) - 1) & 1); }
          // the segment-state products in the S columns have been read
          if (sa >= 1) { MMA_WAIT(kSaFree0 + ((sa - 1) & 1), ((sa - 1) >> 1) & 1); }
          if (sa >= 2) { MMA_WAIT(kSaFree0 + ((sa - 2) & 1), ((sa - 2) >> 1) & 1); }
          issue_cb(it, bt);
          issued = true;
        }
        const uint32_t aC0 = smem_u32(sm.C(st, 0)), aC1 = smem_u32(sm.C(st, 1));
        const uint32_t aX = smem_u32(sm.X(st));
        bool need_cb = inf.idx + 1 < inf.cnt;
        bool need_yo = true, need_yd = true;
        const unsigned long long tw = gtime();
        bool timed_out = false;
        while (need_cb || need_yo || need_yd) {
          bool progressed = false;
          if (need_cb && mbar_test_wait(&bars[kFull0 + ((it + 1) & 1)], ((it + 1) >> 1) & 1) &&
              (bt + 1 < 2 ||
               mbar_test_wait(&bars[kCbEmpty0 + ((bt + 1) & 1)], (((bt + 1) >> 1) - 1) & 1))) {
            tc_fence_after();
            issue_cb(it + 1, bt + 1);
            need_cb = false;
            progressed = true;
          }
          if (need_yo && (bt < 1 || mbar_test_wait(&bars[kYoFree], (bt - 1) & 1)) &&
              mbar_test_wait(&bars[kHFull], bt & 1)) {
            // [Y_off_hi | Y_off_lo] = C [H_hi | H_lo]^T: the two 64-column
            // halves of the B operand are the hi and lo tiles, kTile apart
            tc_fence_after();
            {
              const uint32_t aH = smem_u32(sm.Ht(0));
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t kb = (k & 3) * 32;
                mma_bf16(tmem + kColYO, sdesc_sw128((k < 4 ? aC0 : aC1) + kb, 16, 1024),
                         sdesc_sw128(aH + k * 2048, kTile, 1024), idYO, k > 0);
              }
            }
            mma_commit(&bars[kHEmpty]);
            need_yo = false;
            progressed = true;
          }
          if (need_yd &&
              (bt < 2 || mbar_test_wait(&bars[kYdFree0 + (bt & 1)], ((bt >> 1) - 1) & 1)) &&
              mbar_test_wait(&bars[kSFull0 + (bt & 1)], (bt >> 1) & 1)) {
            // Y_diag = S X, S (hi, lo) read from TMEM: K block k (columns
            // j = 16k .. 16k+15 of S) holds 8 columns of hi pairs, then 8 of
            // lo pairs
            tc_fence_after();
            const uint32_t cbcol = tmem + kColCB + (bt & 1) * 128;
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                mma_bf16_tmem_a(tmem + kColYD + (bt & 1) * 64, cbcol + 16 * k + 8 * part,
                                sdesc_sw128(aX + k * 2048, kTile, 1024), idYD,
                                part > 0 || k > 0);
            need_yd = false;
            progressed = true;
          }
          if (!progressed) {
            if (*abort_v || gtime() - tw > prm.wait_ns) {
              timed_out = true;
              break;
            }
            // nothing ready: sleep on the input that usually comes next
            // rather than spin, so the math warps sharing this warp's
            // scheduler keep its issue slots
            if (need_yd)
              (void)mbar_try_wait_hint(&bars[kSFull0 + (bt & 1)], (bt >> 1) & 1, 200);
            else if (need_yo)
              (void)mbar_try_wait_hint(&bars[kHFull], bt & 1, 200);
            else
              (void)mbar_try_wait_hint(&bars[kFull0 + ((it + 1) & 1)], ((it + 1) >> 1) & 1, 200);
          }
        }
        if (timed_out) {
          fail(SSD_ERR_TIMEOUT);
          break;
        }
        mma_commit(&bars[kAccFull]);
        mma_commit(&bars[kCbEmpty0 + (bt & 1)]);
        mma_commit(&bars[kEmpty0 + st]);
        ++bt;
        ++it;
      }
#undef MMA_WAIT
      if (issued) {
        // every MMA issued must complete before TMEM is released
        mma_commit(&bars[kMmaDone]);
        if (!wait_bar(&bars[kMmaDone], 0, prm.wait_ns)) fail(SSD_ERR_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ math warps
    // Warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 (a warp may only
    // touch its own lane quarter) and takes column quarter cq = w / 4: one
    // 32-column block of the 128 x 128 mask, and columns 16 cq .. 16 cq + 15
    // of every 64-wide (headdim) tile.
    const int wq = warp & 3;
    const int cq = warp >> 2;
    const int r = 32 * wq + lane;  // TMEM lane: token row i / state row n / token j
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    // use counters: ring chunk, forward chunk, w o X buffer, segment-state
    // accumulator, hand-off rendezvous
    uint32_t it = 0, bt = 0, xu = 0, xu1 = 0, sa_m = 0, nhand = 0;
    uint32_t ny = 0;     // epilogues whose staged y this warp has released
    bool ypend = false;  // a y tile staged in the w o X buffer may still be read
    float hreg[16];  // fp32 state H[p][n = r], p = 16 cq + q

    // This warp's arrival number `use` (0, 1, ...) on a barrier that all
    // math warps arrive on.  Arrivals carry no phase, so a warp must never
    // arrive twice before the others arrived once; on every such barrier
    // that holds by construction: between two arrivals a warp waits on a
    // phase that cannot complete before the first arrival's phase did (the
    // tensor core's next use of the buffer, the next TMA fill of the stage,
    // or, for kYRead, the phase itself).
    auto arrive_seq = [&](int bar, uint32_t use) -> bool {
      (void)use;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bar]);
      return true;
    };

    // this thread's decay values of the chunk in stage `stg`: the chunk's
    // total and row r's cumulative log2-decay, and row r's dt (the plain
    // variant) or E-table entry (the fused-epilogue variant)
    auto chunk_vals = [&](int stg, float& c2l, float& c2r, float& er) {
      const float* c2 = sm.c2(stg);
      c2l = c2[kQ - 1];
      c2r = c2[r];
      if constexpr (kEpi)
        er = sm.E(stg)[r];
      else
        er = __bfloat162float(sm.dt(stg)[r]);
    };

    // The decay mask S of forward chunk number `pbt`, written as bf16 hi/lo
    // pairs over its C B^T in TMEM.  Each 16-column block j in [16 k, 16 k +
    // 16) of a row (the MMA's K block k) is rewritten in place as 8 columns
    // of hi pairs followed by 8 columns of lo pairs, so a thread only
    // overwrites TMEM it has just read itself.  This warp owns blocks 2 cq
    // and 2 cq + 1 of its rows.
    auto build_mask = [&](uint32_t pbt, int stg, float c2r, float Dh, bool ez) -> bool {
      const float* c2 = sm.c2(stg);
      if (!wait_bar_warp(&bars[kCbFull0 + (pbt & 1)], (pbt >> 1) & 1, prm.wait_ns)) return false;
      tc_fence_after();
      const uint32_t cbcol = tmem + kColCB + (pbt & 1) * 128 + lane_addr;
      const int b = 32 * wq;   // first row of this warp's lanes
      const int j0 = 32 * cq;  // first column of this warp's two blocks
      if (j0 > b) {
        // strictly above the diagonal: causal zeros
        uint32_t z[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) z[q] = 0u;
        tmem_st16(cbcol + j0, z);
        tmem_st16(cbcol + j0 + 16, z);
      } else if (ez) {
        // S[i][j] = G[i][j] exp(cum_i) E[j], E from the chunk's table
        const float ei = fast_exp2(c2r);
        const float* Et = sm.E(stg);
        const bool diag = j0 == b;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float g[16];
          tmem_ld16(cbcol + j0 + 16 * half, g);
          tmem_ld_wait();
          tie16(g);
          uint32_t pk[16];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int ja = j0 + 16 * half + 4 * m;
            const float4 e4 = *reinterpret_cast<const float4*>(Et + ja);
            float sv[4] = {g[4 * m] * (ei * e4.x), g[4 * m + 1] * (ei * e4.y),
                           g[4 * m + 2] * (ei * e4.z), g[4 * m + 3] * (ei * e4.w)};
            if (diag) {
              // causal; the skip term D x rides on the diagonal: S[i][i] + D
#pragma unroll
              for (int k = 0; k < 4; ++k)
                sv[k] = ja + k < r ? sv[k] : (ja + k == r ? sv[k] + Dh : 0.f);
            }
            split2(sv[0], sv[1], pk[2 * m], pk[8 + 2 * m]);
            split2(sv[2], sv[3], pk[2 * m + 1], pk[8 + 2 * m + 1]);
          }
          tmem_st16(cbcol + j0 + 16 * half, pk);
        }
      } else {
        // exp(cum_i - cum_j) = exp(cum_i - cum_b) exp(cum_b - cum_j): the
        // row factor u is this thread's own, the column factor
        // exp(cum_b - cum_j) dt_j is computed by lane j - j0 and broadcast.
        // Below the diagonal both factors are <= 1.  On the diagonal block
        // the column factor is >= 1, so the factored form is used only when
        // the block's whole decay keeps both inside fp32's range (almost
        // always); otherwise each entry takes its own exponential.
        const float c2b = c2[b];
        const bool diag = j0 == b;
        const bool direct = diag && !(fabsf(c2b - c2[b + 31]) < 120.f);
        if (!direct) {
          const float u = fast_exp2(c2r - c2b);
          // the chunk is not `ez` (in the fused-epilogue variant its E slot holds dt)
          const float dtj = kEpi ? sm.E(stg)[j0 + lane] : __bfloat162float(sm.dt(stg)[j0 + lane]);
          const float vl = fast_exp2(c2b - c2[j0 + lane]) * dtj;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float g[16];
            tmem_ld16(cbcol + j0 + 16 * half, g);
            tmem_ld_wait();
            tie16(g);
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float v0 = __shfl_sync(0xffffffffu, vl, 16 * half + 2 * q);
              const float v1 = __shfl_sync(0xffffffffu, vl, 16 * half + 2 * q + 1);
              float s0 = g[2 * q] * v0 * u, s1 = g[2 * q + 1] * v1 * u;
              if (diag) {
                // causal; the skip term D x rides on the diagonal: S[i][i] + D
                const int ja = j0 + 16 * half + 2 * q;
                s0 = ja < r ? s0 : (ja == r ? s0 + Dh : 0.f);
                s1 = ja + 1 < r ? s1 : (ja + 1 == r ? s1 + Dh : 0.f);
              }
              split2(s0, s1, pk[q], pk[8 + q]);
            }
            tmem_st16(cbcol + j0 + 16 * half, pk);
          }
        } else {
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float g[16];
            tmem_ld16(cbcol + j0 + 16 * half, g);
            tmem_ld_wait();
            tie16(g);
            uint32_t pk[16];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              // keeps the table loads of one group of 4 columns together
              // (hoisting all of them costs registers the warp does not have)
              asm volatile("" ::: "memory");
              const int ja = j0 + 16 * half + 4 * m;
              const float4 cc = *reinterpret_cast<const float4*>(c2 + ja);
              float dd[4];
              if constexpr (kEpi) {
                // the chunk is not `ez`: its E slot holds dt
#pragma unroll
                for (int q = 0; q < 4; ++q) dd[q] = sm.E(stg)[ja + q];
              } else {
                const uint2 db = *reinterpret_cast<const uint2*>(sm.dt(stg) + ja);
                dd[0] = bf_lo(db.x);
                dd[1] = bf_hi(db.x);
                dd[2] = bf_lo(db.y);
                dd[3] = bf_hi(db.y);
              }
              const float s0 = ja <= r ? g[4 * m] * fast_exp2(c2r - cc.x) * dd[0] : 0.f;
              const float s1 = ja + 1 <= r ? g[4 * m + 1] * fast_exp2(c2r - cc.y) * dd[1] : 0.f;
              const float s2 = ja + 2 <= r ? g[4 * m + 2] * fast_exp2(c2r - cc.z) * dd[2] : 0.f;
              const float s3 = ja + 3 <= r ? g[4 * m + 3] * fast_exp2(c2r - cc.w) * dd[3] : 0.f;
              const int dq = r - ja;
              const float d0 = dq == 0 ? Dh : 0.f, d1 = dq == 1 ? Dh : 0.f;
              const float d2 = dq == 2 ? Dh : 0.f, d3 = dq == 3 ? Dh : 0.f;
              split2(s0 + d0, s1 + d1, pk[2 * m], pk[8 + 2 * m]);
              split2(s2 + d2, s3 + d3, pk[2 * m + 1], pk[8 + 2 * m + 1]);
            }
            tmem_st16(cbcol + j0 + 16 * half, pk);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      // one "S ready" barrier per S buffer: the math warps can get a chunk
      // ahead of the MMA (the next C B^T is issued before this S is used),
      // never two
      return arrive_seq(kSFull0 + (pbt & 1), pbt >> 1);
    };

    // w o X (w = weight of row r) of the chunk in stage `stg` as hi/lo bf16
    // pairs, this thread's 16 columns.
    auto compute_xw = [&](int stg, float w, uint32_t (&ph)[8], uint32_t (&pl)[8]) {
      const uint8_t* Xs = sm.X(stg);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 xv = *reinterpret_cast<const uint4*>(Xs + sw128_offset(r, 2 * cq + c));
        split2(w * bf_lo(xv.x), w * bf_hi(xv.x), ph[4 * c + 0], pl[4 * c + 0]);
        split2(w * bf_lo(xv.y), w * bf_hi(xv.y), ph[4 * c + 1], pl[4 * c + 1]);
        split2(w * bf_lo(xv.z), w * bf_hi(xv.z), ph[4 * c + 2], pl[4 * c + 2]);
        split2(w * bf_lo(xv.w), w * bf_hi(xv.w), ph[4 * c + 3], pl[4 * c + 3]);
      }
    };
    // the Xw buffer once the tensor core has read its previous contents
    auto store_xw = [&](const uint32_t (&ph)[8], const uint32_t (&pl)[8]) -> bool {
      if (xu >= 1 && !wait_bar_warp(&bars[kXwEmpty], (xu - 1) & 1, prm.wait_ns)) return false;
      if (ypend) {
        // the buffer also stages the previous chunk's y for its TMA stores:
        // every warp's store must have read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        if (!arrive_seq(kYRead, ny)) return false;
        if (!wait_bar_warp(&bars[kYRead], ny & 1, prm.wait_ns)) return false;
        ++ny;
        ypend = false;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t off = sw128_offset(r, 2 * cq + c);
        *reinterpret_cast<uint4*>(sm.Xw(0) + off) =
            make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
        *reinterpret_cast<uint4*>(sm.Xw(1) + off) =
            make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
      }
      fence_proxy_async_smem();
      if (!arrive_seq(kXwFull, xu)) return false;
      ++xu;
      return true;
    };
    // pass A's second w o X buffer: the H^T tiles, free until the hand-off
    // (the last forward chunk's C H^T has completed: its accumulators were
    // waited for)
    auto store_xw1 = [&](const uint32_t (&ph)[8], const uint32_t (&pl)[8]) -> bool {
      if (xu1 >= 1 && !wait_bar_warp(&bars[kXwEmpty1], (xu1 - 1) & 1, prm.wait_ns)) return false;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t off = sw128_offset(r, 2 * cq + c);
        *reinterpret_cast<uint4*>(sm.Ht(0) + off) =
            make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
        *reinterpret_cast<uint4*>(sm.Ht(1) + off) =
            make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
      }
      fence_proxy_async_smem();
      if (!arrive_seq(kXwFull1, xu1)) return false;
      ++xu1;
      return true;
    };
    // the math warps are done reading the stage of ring chunk `pit`
    auto release_stage = [&](uint32_t pit) -> bool {
      return arrive_seq(kEmpty0 + (pit & 1), pit >> 1);
    };
    // H^T (hi, lo) for C H^T: row n = r, this thread's 16 columns p
    auto store_ht = [&]() {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint4 h4, l4;
        split2(hreg[8 * c + 0], hreg[8 * c + 1], h4.x, l4.x);
        split2(hreg[8 * c + 2], hreg[8 * c + 3], h4.y, l4.y);
        split2(hreg[8 * c + 4], hreg[8 * c + 5], h4.z, l4.z);
        split2(hreg[8 * c + 6], hreg[8 * c + 7], h4.w, l4.w);
        const uint32_t off = sw128_offset(r, 2 * cq + c);
        *reinterpret_cast<uint4*>(sm.Ht(0) + off) = h4;
        *reinterpret_cast<uint4*>(sm.Ht(1) + off) = l4;
      }
      fence_proxy_async_smem();
    };

#define MATH_TRY(expr)     \
  if (!(expr)) {           \
    fail(SSD_ERR_TIMEOUT); \
    goto math_done;        \
  }
    while (true) {
      MATH_TRY(wait_bar_warp(&bars[kFull0 + (it & 1)], (it >> 1) & 1, prm.wait_ns));
      const TileInfo* u0p = sm.info(it & 1);
      if (u0p->kind == kKindEnd || __any_sync(0xffffffffu, *abort_v)) break;
      const int h = u0p->h;
      const int nA = u0p->nA;
      const int u_unit = u0p->unit, u_sigma = u0p->sigma, u_s = u0p->s;
      const int u_last = u0p->last_seg;
      const float Dh = prm.D ? prm.D[h] : 0.f;
      // the initial state of a sequence's first segment is loaded now so its
      // latency hides behind the segment-state pass
      if (u_sigma == 0) {
        const float* ini = prm.init ? prm.init + ((long long)u_s * prm.H + h) * kPN : nullptr;
#pragma unroll
        for (int q = 0; q < 16; ++q) hreg[q] = ini ? __ldg(ini + (16 * cq + q) * kN + r) : 0.f;
      }

      // -------- pass A: the segment's chunk states, chunks walked backwards.
      // Each chunk's state S_c (B^T (w o X) with the chunk-local weights w_j
      // = exp(cum_last - cum_j) dt_j) is read back from TMEM, kept in this
      // CTA's scratch (global memory, L2-resident; each thread reloads only
      // what it stored) for the forward pass, and folded into the segment-
      // local state H_loc = sum_c exp(sum of the later chunks' dt A) S_c.
      float hloc[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) hloc[q] = 0.f;
      float later = 0.f;  // sum of the log2-decays of the chunks folded so far
      float* stb = prm.stbuf + (long long)blockIdx.x * kStSlots * kPN + (16 * cq) * kN + r;
      // fold pass-A chunk `kk` (its product is in S-column buffer `sa_m & 1`)
      auto fold = [&](int kk, float c2l_kk) -> bool {
        if (!wait_bar_warp(&bars[kSaFull0 + (sa_m & 1)], (sa_m >> 1) & 1, prm.wait_ns)) return false;
        tc_fence_after();
        float hi[16], lo[16];
        const uint32_t col = tmem + kColSA + (sa_m & 1) * 128 + lane_addr + 16 * cq;
        tmem_ld16(col, hi);
        tmem_ld16(col + 64, lo);
        tmem_ld_wait();
        tie16(hi);
        tie16(lo);
        tc_fence_before();
        if (!arrive_seq(kSaFree0 + (sa_m & 1), sa_m >> 1)) return false;
        ++sa_m;
        const float wl = fast_exp2(later);
        float* dst = stb + (long long)(nA - 1 - kk) * kPN;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float sc = hi[q] + lo[q];
          __stcg(dst + q * kN, sc);
          hloc[q] += wl * sc;
        }
        later += c2l_kk;
        return true;
      };
      float c2l_prev = 0.f;
      for (int k = 0; k < nA; ++k) {
        if (k > 0) MATH_TRY(wait_bar_warp(&bars[kFull0 + (it & 1)], (it >> 1) & 1, prm.wait_ns));
        float c2l, c2r, er;
        chunk_vals(it & 1, c2l, c2r, er);
        uint32_t ph[8], pl[8];
        // w_r = exp(cum_last - cum_r) dt_r, from E (= exp(-cum_r) dt_r) when
        // the chunk's table holds it, else from dt_r
        float wr;
        if constexpr (kEpi)
          wr = fast_exp2(c2l - (sm.info(it & 1)->ez ? 0.f : c2r)) * er;
        else
          wr = fast_exp2(c2l - c2r) * er;
        compute_xw(it & 1, wr, ph, pl);
        MATH_TRY(release_stage(it));
        if ((k & 1) == 0) {
          MATH_TRY(store_xw(ph, pl));
        } else {
          MATH_TRY(store_xw1(ph, pl));
        }
        // the previous chunk's product, read while this one's is computed
        if (k > 0) MATH_TRY(fold(k - 1, c2l_prev));
        c2l_prev = c2l;
        ++it;
      }
      if (nA > 0) MATH_TRY(fold(nA - 1, c2l_prev));

      // -------- segment hand-off
      if (u_sigma != 0) {
        const int pred = u_unit - prm.H;  // same sequence and head, previous segment
        if (tid == 0) {
          const unsigned long long t0 = gtime();
          while (ld_acquire(prm.flags + pred) == 0) {
            if (gtime() - t0 > prm.wait_ns) {
              fail(SSD_ERR_TIMEOUT);
              break;
            }
          }
        }
        MATH_TRY(math_sync(&bars[kSyncHand], nhand & 1, prm.wait_ns));
        ++nhand;
        if (__any_sync(0xffffffffu, *abort_v)) goto math_done;
        const float* src = prm.slots + (long long)pred * kPN;
#pragma unroll
        for (int q = 0; q < 16; ++q) hreg[q] = __ldcg(src + (16 * cq + q) * kN + r);
      }
      if (!u_last) {
        // this segment's end state exp(sum dt A) H_in + H_loc; the release
        // flag follows once the first forward chunk is queued
        const float aseg = fast_exp2(later);
        float* dst = prm.slots + (long long)u_unit * kPN;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          __stcg(dst + (16 * cq + q) * kN + r, aseg * hreg[q] + hloc[q]);
      }
      // the running state H_in, split into bf16 hi/lo, to the B operand of C H^T
      if (bt >= 1) MATH_TRY(wait_bar_warp(&bars[kHEmpty], (bt - 1) & 1, prm.wait_ns));
      store_ht();
      MATH_TRY(arrive_seq(kHFull, bt));

      // -------- pass B: the forward over the segment's chunks from H_in.
      // Chunk t's mask is built two chunks ahead (at the end of iteration
      // t - 2).  The values of a chunk needed after its stage is handed back
      // (first token, length, decay, exp(cum)) are kept in registers; its
      // state product comes from the scratch the segment-state pass filled.
      {
        MATH_TRY(wait_bar_warp(&bars[kFull0 + (it & 1)], (it >> 1) & 1, prm.wait_ns));
        const TileInfo* ci = sm.info(it & 1);
        const int nB = ci->cnt;
        const int s_seq = ci->s, last_seg = ci->last_seg;
        long long t0_cur = ci->t0;
        int len_cur = ci->len;
        float a_cur, ei_cur;
        {
          float c2l, c2r, er;
          chunk_vals(it & 1, c2l, c2r, er);
          a_cur = fast_exp2(c2l);
          ei_cur = fast_exp2(c2r);
          MATH_TRY(build_mask(bt, it & 1, c2r, Dh, sm.info(it & 1)->ez != 0));
          MATH_TRY(release_stage(it));
        }
        if (!u_last) {
          __threadfence();
          MATH_TRY(math_sync(&bars[kSyncHand], nhand & 1, prm.wait_ns));
          ++nhand;
          if (tid == 0 && u_unit != prm.hold_unit) st_release(prm.flags + u_unit, 1);
        }
        if (nB > 1) {
          MATH_TRY(wait_bar_warp(&bars[kFull0 + ((it + 1) & 1)], ((it + 1) >> 1) & 1, prm.wait_ns));
          float c2l, c2r, er;
          chunk_vals((it + 1) & 1, c2l, c2r, er);
          MATH_TRY(build_mask(bt + 1, (it + 1) & 1, c2r, Dh, sm.info((it + 1) & 1)->ez != 0));
        }
        long long t0_nxt = 0;
        int len_nxt = 0;
        float a_nxt = 0.f, ei_nxt = 0.f;
        for (int t = 0; t < nB; ++t) {
          const bool more = t + 1 < nB;
          // this chunk's state product, from the segment-state pass (loaded
          // first: its latency hides behind the wait for the accumulators)
          float sv[16];
          {
            const float* srcs = stb + (long long)t * kPN;
#pragma unroll
            for (int q = 0; q < 16; ++q) sv[q] = __ldcg(srcs + q * kN);
          }
          // the gate values of this thread's 16 outputs (epilogue variant)
          uint4 zv[2];
          if constexpr (kEpi) {
            if (ep.z && r < len_cur) {
              const uint4* zs = reinterpret_cast<const uint4*>(
                  ep.z + (t0_cur + r) * ((long long)prm.H * kP) + h * kP + 16 * cq);
              zv[0] = __ldg(zs);
              zv[1] = __ldg(zs + 1);
            } else {
              zv[0] = make_uint4(0u, 0u, 0u, 0u);
              zv[1] = zv[0];
            }
          }
          // this chunk's accumulators
          MATH_TRY(wait_bar_warp(&bars[kAccFull], bt & 1, prm.wait_ns));
          tc_fence_after();
          const float ei = ei_cur;
          float* yrow = prm.y + ((t0_cur + r) * prm.H + h) * kP + 16 * cq;
          // y = Y_diag + exp(cum_i) (Y_off_hi + Y_off_lo), 8 columns (D x is
          // part of Y_diag: D sits on the diagonal of S).
          // A warp whose 32 rows are all valid stages its 32 x 16 tile in
          // the w o X buffer (unused during a forward pass; 64B-swizzled
          // fp32 rows, 2 KB per warp, each warp its own; or plain 32-byte
          // rows of a bf16 y) and writes it with one TMA store; rows of a
          // ragged last chunk are stored directly.
          const bool tma_y = 32 * wq + 32 <= len_cur;
          uint8_t* ytile = sm.Xw(0) + warp * 2048;
          if (tma_y) {
            // this warp's previous tile must have been read by its store
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
          auto emit_y = [&](int half, const float (&yd)[8], const float (&yh)[8],
                            const float (&yl)[8]) {
            float o[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) o[c] = yd[c] + ei * (yh[c] + yl[c]);
            if constexpr (kEpi) {
              if (ep.z) {
                // gate: y * silu(z) = y * z / (1 + exp(-z))
                const uint32_t zw[4] = {zv[half].x, zv[half].y, zv[half].z, zv[half].w};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const float zc = (c & 1) ? bf_hi(zw[c >> 1]) : bf_lo(zw[c >> 1]);
                  o[c] *= zc / (1.f + fast_exp2(-zc * kLog2e));
                }
              }
              if (ep.y_bf16) {
                uint4 w;
                w.x = pack_bf16(o[0], o[1]);
                w.y = pack_bf16(o[2], o[3]);
                w.z = pack_bf16(o[4], o[5]);
                w.w = pack_bf16(o[6], o[7]);
                if (tma_y) {
                  *reinterpret_cast<uint4*>(ytile + lane * 32 + 16 * half) = w;
                } else if (r < len_cur) {
                  __stcs(reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(prm.y) +
                                                  ((t0_cur + r) * prm.H + h) * kP + 16 * cq) + half, w);
                }
                return;
              }
            }
            if (tma_y) {
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int chunk = 2 * half + c;
                *reinterpret_cast<float4*>(ytile + lane * 64 + 16 * (chunk ^ ((lane >> 1) & 3))) =
                    make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
              }
            } else if (r < len_cur) {
              if (prm.y_v8) {
                st_global_cs_v8(yrow + 8 * half, o);
              } else {
                __stcs(reinterpret_cast<float4*>(yrow + 8 * half), make_float4(o[0], o[1], o[2], o[3]));
                __stcs(reinterpret_cast<float4*>(yrow + 8 * half + 4), make_float4(o[4], o[5], o[6], o[7]));
              }
            }
          };
          // the state (it feeds the next chunk's C H^T)
#pragma unroll
          for (int q = 0; q < 16; ++q) hreg[q] = a_cur * hreg[q] + sv[q];
          // this chunk state's lines are dead now (each 128-byte line is one
          // p row of this warp's 32 n): drop them from L2 unwritten, so the
          // scratch never costs DRAM write bandwidth
          __syncwarp();
          if (lane < 16) discard_l2_line(stb - lane + (long long)t * kPN + lane * kN);
          if (more) {
            MATH_TRY(wait_bar_warp(&bars[kHEmpty], bt & 1, prm.wait_ns));
            store_ht();
            MATH_TRY(arrive_seq(kHFull, bt + 1));
          } else if (last_seg && prm.final_states) {
            float* fin = prm.final_states + ((long long)s_seq * prm.H + h) * kPN;
#pragma unroll
            for (int q = 0; q < 16; ++q) fin[(16 * cq + q) * kN + r] = hreg[q];
          }
          {
            float yd[8], yh[8], yl[8];
            tmem_ld8(tmem + kColYD + (bt & 1) * 64 + lane_addr + 16 * cq, yd);
            tmem_ld8(tmem + kColYO + lane_addr + 16 * cq, yh);
            tmem_ld8(tmem + kColYO + lane_addr + 64 + 16 * cq, yl);
            tmem_ld_wait();
            tie8(yd);
            tie8(yh);
            tie8(yl);
            emit_y(0, yd, yh, yl);
          }
          {
            float yd[8], yh[8], yl[8];
            tmem_ld8(tmem + kColYD + (bt & 1) * 64 + lane_addr + 16 * cq + 8, yd);
            tmem_ld8(tmem + kColYO + lane_addr + 16 * cq + 8, yh);
            tmem_ld8(tmem + kColYO + lane_addr + 64 + 16 * cq + 8, yl);
            tmem_ld_wait();
            tie8(yd);
            tie8(yh);
            tie8(yl);
            tc_fence_before();
            MATH_TRY(arrive_seq(kYoFree, bt));
            MATH_TRY(arrive_seq(kYdFree0 + (bt & 1), bt >> 1));
            emit_y(1, yd, yh, yl);
          }
          if (tma_y) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&map_y, ytile, h * kP + 16 * cq, (int)(t0_cur + 32 * wq));
              bulk_commit();
            }
          }
          ypend = true;
          if (more) {
            // chunk t+1 (its stage is still held; its mask is built): its
            // values, then the stage goes back to the producer
            const TileInfo* ni = sm.info((it + 1) & 1);
            t0_nxt = ni->t0;
            len_nxt = ni->len;
            float c2l, c2r, er;
            chunk_vals((it + 1) & 1, c2l, c2r, er);
            a_nxt = fast_exp2(c2l);
            ei_nxt = fast_exp2(c2r);
            MATH_TRY(release_stage(it + 1));
          }
          if (t + 2 < nB) {
            // chunk t+2's mask, in the stage chunk t has handed back
            MATH_TRY(wait_bar_warp(&bars[kFull0 + ((it + 2) & 1)], ((it + 2) >> 1) & 1, prm.wait_ns));
            float c2l, c2r, er;
            chunk_vals((it + 2) & 1, c2l, c2r, er);
            MATH_TRY(build_mask(bt + 2, (it + 2) & 1, c2r, Dh, sm.info((it + 2) & 1)->ez != 0));
          }
          ++bt;
          ++it;
          t0_cur = t0_nxt;
          len_cur = len_nxt;
          a_cur = a_nxt;
          ei_cur = ei_nxt;
        }
      }
    }
  math_done:
    // y tiles still being written must land before the CTA exits
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
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

bool tc_supported(const FwdArgs& a) {
  return a.dtype == SSD_DT_BF16 && a.P == kP && a.N == kN;
}

size_t tc_workspace_bytes(const FwdArgs& a) { return ws_layout(a).total; }

ssd_status_t tc_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit) {
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
  CUtensorMap mx, mb, mc, my, mz;
  const bool work = ntok > 0 && mu > 0;
  const bool epi = a.z != nullptr || a.y_bf16 || a.dt_softplus;
  if (work && (!tc_make_map_bf16(&mx, a.x, ntok, (long long)a.H * kP) ||
               !tc_make_map_bf16(&mb, a.B, ntok, (long long)a.G * kN) ||
               !tc_make_map_bf16(&mc, a.C, ntok, (long long)a.G * kN) ||
               (a.y_bf16 ? !tc_make_map_y_bf16(&my, a.y, ntok, (long long)a.H * kP)
                         : !tc_make_map_y_f32(&my, a.y, ntok, (long long)a.H * kP)) ||
               // z is only prefetched through its map (x stands in when absent)
               !tc_make_map_bf16(&mz, a.z ? a.z : a.x, ntok, (long long)a.H * kP)))
    return SSD_ERR_CUDA;
  Params p;
  p.dt = static_cast<const __nv_bfloat16*>(a.dt);
  p.A = a.A;
  p.D = a.D;
  p.init = a.init;
  p.y = a.y;
  p.final_states = a.final_states;
  EpiParams ep;
  ep.dt_bias = a.dt_bias;
  ep.dt_softplus = a.dt_softplus;
  ep.z = static_cast<const __nv_bfloat16*>(a.z);
  ep.y_bf16 = a.y_bf16;
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
    attr_err = cudaFuncSetAttribute(ssd_tc_fwd_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(ssd_tc_fwd_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
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
  const cudaError_t le =
      epi ? cudaLaunchKernelEx(&cfg, ssd_tc_fwd_kernel<true>, mx, mb, mc, my, mz, p, ep)
          : cudaLaunchKernelEx(&cfg, ssd_tc_fwd_kernel<false>, mx, mb, mc, my, mz, p, ep);
  if (le != cudaSuccess) return SSD_ERR_CUDA;
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
