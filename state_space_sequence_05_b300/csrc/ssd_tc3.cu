// ssd_tc3.cu -- tcgen05 tensor-core SSD forward for bf16 inputs, headdim 64,
// dstate 128 (the Mamba-2 2.7B layer shape), as three kernels.
//
// It evaluates the SSD chunked algorithm ("Transformers are SSMs Review",
// sec. 3-2 (4)) with 128-token chunks.  Each sequence is cut into segments
// of a few chunks and a work unit is one (sequence, segment, head).  The
// four steps of the algorithm are split the way the review's sec. 3-2 (6)
// splits a sequence across devices: only the states at segment boundaries
// pass between the pieces.
//
//   1. Segment states (ssd_seg_state_kernel).  Per unit, the state the
//      segment leaves from a zero state,
//        H_loc = sum_j exp(cum_end - cum_j) dt_j x_j B_j^T   (j over the segment),
//      as one tensor-core product B^T (w o X) accumulated over the
//      segment's chunks, and the segment's total log2-decay.
//   2. State passing (ssd_seg_pass_kernel).  Per (sequence, head), the
//      recurrence over segments H_in(s + 1) = exp(decay_s) H_in(s) + H_loc(s)
//      from the initial state, elementwise (the composition of affine maps
//      (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2), "Mamba ... review",
//      feghi.github.io, sec. 4); the state after the last segment is the
//      final state.
//   3. Outputs (ssd_seg_out_kernel).  Per unit, from H_in, chunk by chunk,
//      with cum_i = sum_{k<=i} dt_k A_h (chunk-local) and the row factor
//      f_i = exp(max(cum_i, -60 ln 2)):
//        G        = C B^T                                (128 x 128, K = dstate)
//        S'[i,j]  = G[i,j] exp(cum_i - cum_j) dt_j / f_i   for j <= i, else 0
//                   (+ D_h / f_i on the diagonal: the skip term D x)
//        y_i      = f_i (S' X + C H_c^T)_i
//        S_c      = B^T (w o X),  w_j = exp(cum_last - cum_j) dt_j
//        H_{c+1}  = exp(cum_last) H_c + S_c
//      so the intra-chunk quadratic form and the off-diagonal term share one
//      accumulator.  For a row decayed less than 2^-60 from the chunk start,
//      S'[i,j] = G[i,j] E_j with the per-chunk table E_j = exp(-cum_j) dt_j
//      (below 2^60 dt_j for every j <= i); a deeper row takes f_i = 2^-60 and
//      its own exponentials, and its state term is scaled by 2^-60 instead of
//      exp(cum_i) < 2^-60 (an absolute change below 2^-60 |C_i H^T|).
//
// No kernel waits on another CTA: the units of kernels 1 and 3 are
// independent, and kernel 2 is elementwise.
//
// Precision: x, B and C are bf16 and used as they are.  The derived fp32
// operands S', w o X and H are each split into bf16 hi (v truncated) and lo
// ((v - hi) truncated), |v - hi - lo| < 2^-14 |v|, both multiplied into fp32
// accumulators (a single bf16 rounding of any of them costs 2-4e-2 of
// RMS(y) in max error on the 2.7B layer).  The hi and lo halves of w o X
// and of H are the two 64-column halves of one N = 128 operand.
//
// Kernels 1 and 3 are persistent (one CTA per SM) with warp roles:
//   warp 16    producer: TMA loads (128-byte swizzle) and the chunk's
//              decay tables;
//   warp 17    MMA issuer (the whole warp; one elected lane issues);
//   warps 0-15 CUDA-core math: tensor-memory lane quarter w % 4, column
//              quarter w / 4.
// Every wait is bounded; on expiry the kernel records SSD_ERR_TIMEOUT and
// unwinds with its tensor memory freed.
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
constexpr int kThreads = 576;
constexpr uint32_t kTile = 16384;  // 128 rows x 128 bytes (bf16)
constexpr uint64_t kT16 = kTile >> 4;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kDeep = -60.f;  // log2 of the smallest row factor

enum : int { kKindChunk = 0, kKindEnd = 1 };

// What the producer tells the other roles about the chunk in a slot.
struct TileInfo {
  long long t0;   // first token of the chunk
  int unit;       // work unit
  int h;          // head
  int len;        // valid rows (1..128)
  int kind;       // kKindChunk or kKindEnd (no more work)
  int first;      // first chunk of its unit in the order walked
  int last;       // last chunk of its unit in the order walked
  int next_unit;  // the unit the producer took next (-1: none), on a last chunk
  float D;        // skip coefficient D_h of the head (0 without D)
  int pad[6];
};
static_assert(sizeof(TileInfo) == 64, "tile info slot");

// A work unit: sequence s, segment sigma, head h (ticket order).
struct Unit {
  long long b, e;  // token range of the sequence
  int u, s, h, g, sigma, tb, te, n;
  int c0;          // global index of the sequence's first chunk
  float D;         // skip coefficient of the head (output kernel)
};

struct UnitPlan {
  const int32_t* uoff;  // [nseq + 2]: unit offsets per sequence, then plan status
  const int32_t* coff;  // [nseq + 1]: chunk offsets per sequence
  SeqInfo si;
  int H, G, seg;
  __device__ __forceinline__ void decode(int v, Unit& X) const {
    const int nseq = si.nseq;
    X.u = v;
    X.s = upper_index(uoff, nseq, v);
    const int rem = v - uoff[X.s];
    X.sigma = rem / H;
    X.h = rem % H;
    X.g = (int)((long long)X.h * G / H);
    X.c0 = coff[X.s];
    X.b = si.begin(X.s);
    X.e = si.end(X.s);
    const int nt = (int)((X.e - X.b + kQ - 1) / kQ);
    X.tb = X.sigma * seg;
    X.te = min(nt, X.tb + seg);
    X.n = X.te - X.tb;
  }
};

// Chunk-local cumulative log2-decay of a chunk from its dt (lane l owns
// tokens 4l .. 4l+3; dt is 0 past the valid rows, so c2 stays flat there).
// Writes c2[128], dt[128] and, when E is given, E[j] = exp2(-c2_j) dt_j.
__device__ __forceinline__ void decay_tables(const __nv_bfloat16 (&d)[4], int len, float A2,
                                             float* c2t, float* Et, __nv_bfloat16* dtt,
                                             int lane) {
  float dv[4], pre[4], run = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    dv[q] = __bfloat162float(d[q]);
    run += dv[q] * A2;
    pre[q] = run;
  }
  float incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float tv = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += tv;
  }
  const float excl = incl - run;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float cq2 = excl + pre[q];
    c2t[4 * lane + q] = cq2;
    if (Et) Et[4 * lane + q] = 4 * lane + q < len ? fast_exp2(-cq2) * dv[q] : 0.f;
    dtt[4 * lane + q] = d[q];
  }
}

// Decay tables of one (chunk, head), as the kernels keep them in shared
// memory: c2 fp32[128], E fp32[128], dt bf16[128].
constexpr uint32_t kTabBytes = 512 + 512 + 256;

// One block per (chunk, tile of 8 heads): the tile's dt read row by row
// (16-byte runs) into shared memory transposed, then one warp per head writes
// its decay tables into tabs[(global chunk) H + h], so that the persistent
// kernels fetch them with one bulk copy per chunk.
constexpr int kTabHeads = 8;
constexpr int kTabRow = kQ + 8;  // padded row of the transposed dt tile
__global__ void __launch_bounds__(256)
    ssd_chunk_tables_kernel(const int32_t* uoff, const int32_t* coff, SeqInfo si, int H,
                            const __nv_bfloat16* dt, const float* A, uint8_t* tabs) {
  __shared__ __align__(16) __nv_bfloat16 dts[kTabHeads * kTabRow];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int nseq = si.nseq;
  if (uoff[nseq + 1] != 0) return;
  const int gc = blockIdx.x;
  if (gc >= coff[nseq]) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = upper_index(coff, nseq, gc);
  const long long t0 = si.begin(s) + (long long)(gc - coff[s]) * kQ;
  const int len = (int)min((long long)kQ, si.end(s) - t0);
  {
    const int h0 = blockIdx.y * kTabHeads;
    const int nh = min(kTabHeads, H - h0);
    for (int e = threadIdx.x; e < kQ * nh; e += blockDim.x) {
      const int j = e / nh, hh = e % nh;
      dts[hh * kTabRow + j] = j < len ? dt[(t0 + j) * H + h0 + hh] : __float2bfloat16(0.f);
    }
    __syncthreads();
    for (int hh = warp; hh < nh; hh += blockDim.x >> 5) {
      const uint2 v = *reinterpret_cast<const uint2*>(dts + hh * kTabRow + 4 * lane);
      __nv_bfloat16 d[4];
      d[0] = __ushort_as_bfloat16((unsigned short)(v.x & 0xffffu));
      d[1] = __ushort_as_bfloat16((unsigned short)(v.x >> 16));
      d[2] = __ushort_as_bfloat16((unsigned short)(v.y & 0xffffu));
      d[3] = __ushort_as_bfloat16((unsigned short)(v.y >> 16));
      const int h = h0 + hh;
      uint8_t* tb = tabs + ((long long)gc * H + h) * kTabBytes;
      decay_tables(d, len, A[h] * kLog2e, reinterpret_cast<float*>(tb),
                   reinterpret_cast<float*>(tb + 512), reinterpret_cast<__nv_bfloat16*>(tb + 1024),
                   lane);
    }
  }
}

// One 16-byte work item of w o X (items k = 0..1023: 8 values of row j =
// k / 8 of the 128B-swizzled x tile), weight w_j = exp2(wl - c2_j) dt_j,
// written as bf16 hi and lo tiles at `dst` (lo one tile after hi).
__device__ __forceinline__ void wx_item(const uint8_t* xt, const float* c2t,
                                        const __nv_bfloat16* dtt, int k, float wl, uint8_t* dst) {
  const int j = k >> 3, c = k & 7;
  const uint32_t off = sw128_offset(j, c);
  const uint4 xv = *reinterpret_cast<const uint4*>(xt + off);
  const float w = fast_exp2(wl - c2t[j]) * __bfloat162float(dtt[j]);
  const f2 ww{w, w};
  uint4 hi, lo;
  split2p(mul2(bf2(xv.x), ww), hi.x, lo.x);
  split2p(mul2(bf2(xv.y), ww), hi.y, lo.y);
  split2p(mul2(bf2(xv.z), ww), hi.z, lo.z);
  split2p(mul2(bf2(xv.w), ww), hi.w, lo.w);
  *reinterpret_cast<uint4*>(dst + off) = hi;
  *reinterpret_cast<uint4*>(dst + kTile + off) = lo;
}

// Chunk states: B^T (MN-major, M = n) times [w o X hi | lo] (MN-major, N = 128).
constexpr uint32_t kIdSt = idesc_bf16(128, 128, true, true);
// C B^T: C and B both K-major.
constexpr uint32_t kIdG = idesc_bf16(128, 128, false, false);
// C (K-major) times [H_hi | H_lo]^T (MN-major, N = 128).
constexpr uint32_t kIdCH = idesc_bf16(128, 128, false, true);
// S' (tensor memory) times X (MN-major, N = 64).
constexpr uint32_t kIdSX = idesc_bf16(128, 64, false, true);

// ============================================================== kernel 1
namespace k1 {
constexpr int kStages = 3;
// A stage: the x tile (overwritten in place by w o X hi), w o X lo, B (n 0..63),
// B (n 64..127).  [hi | lo] is the N = 128 operand of the state product.
constexpr uint32_t kStageBytes = 4 * kTile;
constexpr uint32_t kOffTabs = kStages * kStageBytes;  // per stage: the chunk's decay tables
constexpr uint32_t kOffInfo = kOffTabs + kStages * kTabBytes;
constexpr uint32_t kOffBars = kOffInfo + kStages * 64;
constexpr uint32_t kBarBytes = 16 * 8;
constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 16;
static_assert(kSmemBytes <= 232448, "shared memory per block");
constexpr uint32_t kTmemCols = 256;  // two accumulators [hi | lo] x 128 columns

enum {
  kFull0 = 0, kFull1, kFull2,          // stage loaded (TMA: tiles and tables)
  kEmpty0 = 3, kEmpty1, kEmpty2,       // stage's state product done (MMA commit)
  kWxFull0 = 6, kWxFull1, kWxFull2,    // w o X written in the stage (math warps)
  kAccFull0 = 9, kAccFull1,            // unit's product complete (MMA commit)
  kAccFree0 = 11, kAccFree1,           // unit's product read (math warps)
  kMmaDone = 13,
  kNumBars
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

struct Params {
  UnitPlan up;
  const uint8_t* tabs;  // per (global chunk, head): decay tables
  float* slots;  // per unit: H_loc [P][N] fp32
  float* dec;    // per unit: total log2-decay of the segment
  int* ticket;   // ticket[0]: work ticket; ticket[1]: line of the first expired wait
  int32_t* status;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
    ssd_seg_state_kernel(const __grid_constant__ CUtensorMap map_x,
                         const __grid_constant__ CUtensorMap map_b, Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (tid == 0) report(prm.status, SSD_ERR_UNSUPPORTED);
    return;
  }
  uint8_t* const sb = smem_raw;
  auto X = [&](int st) { return sb + st * kStageBytes; };
  auto Bt = [&](int st) { return sb + st * kStageBytes + 2 * kTile; };
  auto c2 = [&](int st) { return reinterpret_cast<float*>(sb + kOffTabs + st * kTabBytes); };
  auto dtt = [&](int st) {
    return reinterpret_cast<__nv_bfloat16*>(sb + kOffTabs + st * kTabBytes + 1024);
  };
  auto info = [&](int st) { return reinterpret_cast<TileInfo*>(sb + kOffInfo) + st; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kOffBars);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(sb + kOffBars + kBarBytes);
  int* abort_p = reinterpret_cast<int*>(sb + kOffBars + kBarBytes + 4);
  const unsigned long long wns = prm.wait_ns;

  if (tid == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(&bars[kFull0 + b], 1);   // expect-tx arrival (tiles, tables)
      mbar_init(&bars[kEmpty0 + b], 1);  // MMA commit
      mbar_init(&bars[kWxFull0 + b], kMathWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kAccFull0 + b], 1);
      mbar_init(&bars[kAccFree0 + b], kMathWarps);
    }
    mbar_init(&bars[kMmaDone], 1);
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

  // the plan's results (unit offsets, tickets) are ready past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the state-passing kernel may be scheduled now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;");
  const int nseq = prm.up.si.nseq;
  const int nunits = prm.up.uoff[nseq];
  const bool plan_ok = prm.up.uoff[nseq + 1] == 0;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Units by ticket; a unit's chunks from the last to the first (the
    // weights need the decay of the later chunks).
    if (lane == 0) {
      prefetch_tmap(&map_x);
      prefetch_tmap(&map_b);
    }
    uint32_t it = 0;
    bool ok = true;
    Unit U;
    auto draw = [&](Unit& Xu) -> bool {
      int v = 0;
      if (lane == 0) v = atomicAdd(prm.ticket, 1);
      v = __shfl_sync(0xffffffffu, v, 0);
      if (v >= nunits) return false;
      prm.up.decode(v, Xu);
      return true;
    };
    // chunk k of unit X in the order walked (the last one first)
    auto coords = [&](const Unit& Xu, int k, long long& t0, int& len) {
      t0 = Xu.b + (long long)(Xu.te - 1 - k) * kQ;
      len = (int)min((long long)kQ, Xu.e - t0);
    };
    bool have = plan_ok && draw(U);
    int k = 0;
    while (have) {
      const Unit C = U;
      const int kc = k;
      long long t0;
      int len;
      coords(C, kc, t0, len);
      if (++k >= U.n) {
        k = 0;
        have = draw(U);
      }
      const int st = (int)(it % kStages);
      if (it >= kStages &&
          !wait_bar_warp(&bars[kEmpty0 + st], ((it / kStages) - 1) & 1u, wns)) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, *abort_v)) { ok = false; break; }
      if (lane == 0) {
        uint64_t* fb = &bars[kFull0 + st];
        TileInfo* inf = info(st);
        inf->t0 = t0;
        inf->unit = C.u;
        inf->h = C.h;
        inf->len = len;
        inf->kind = kKindChunk;
        inf->first = kc == 0;
        inf->last = kc == C.n - 1;
        inf->next_unit = -1;
        const int gc = C.c0 + (C.te - 1 - kc);
        mbar_arrive_expect_tx(fb, 3 * kTile + kTabBytes);
        tma_load_2d(X(st), &map_x, fb, C.h * kP, (int)t0);
        tma_load_2d(Bt(st), &map_b, fb, C.g * kN, (int)t0);
        tma_load_2d(Bt(st) + kTile, &map_b, fb, C.g * kN + 64, (int)t0);
        bulk_load(c2(st), prm.tabs + ((long long)gc * prm.up.H + C.h) * kTabBytes, kTabBytes, fb);
        if (have) {
          long long nt0;
          int nlen;
          coords(U, k, nt0, nlen);
          tma_prefetch_2d(&map_x, U.h * kP, (int)nt0);
        }
      }
      __syncwarp();
      ++it;
    }
    const int st = (int)(it % kStages);
    if (ok && (it < kStages ||
               wait_bar_warp(&bars[kEmpty0 + st], ((it / kStages) - 1) & 1u, wns))) {
      if (lane == 0) {
        info(st)->kind = kKindEnd;
        mbar_arrive(&bars[kFull0 + st]);
      }
    } else if (lane == 0) {
      if (ok) fail(SSD_ERR_TIMEOUT);
      // aborting: loads still in flight must land before the CTA may exit
      for (uint32_t q = (it >= kStages ? it - kStages : 0); q < it; ++q)
        (void)wait_bar(&bars[kFull0 + q % kStages], (q / kStages) & 1u, wns);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint64_t dBt0 = sdesc_sw128(smem_u32(Bt(0)), kTile, 1024);  // MN-major B^T
    const uint64_t dW0 = sdesc_sw128(smem_u32(X(0)), kTile, 1024);    // [w o X hi | lo]
    constexpr uint64_t kSt16 = kStageBytes >> 4;
    uint32_t it = 0, uc = 0;
    bool issued = false;
#define MMA_WAIT(bar, par)                      \
  if (!wait_bar_warp(&bars[bar], (par), wns)) { \
    if (lane == 0) fail(SSD_ERR_TIMEOUT);       \
    goto mma_done;                              \
  }
    while (true) {
      const int st = (int)(it % kStages);
      MMA_WAIT(kFull0 + st, (it / kStages) & 1u);
      const TileInfo inf = *info(st);
      if (inf.kind == kKindEnd || *abort_v) break;
      MMA_WAIT(kWxFull0 + st, (it / kStages) & 1u);
      const int ab = uc & 1;
      if (inf.first && uc >= 2) { MMA_WAIT(kAccFree0 + ab, ((uc >> 1) - 1) & 1u); }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t d = tmem + ab * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(d, dBt0 + st * kSt16 + kk * 128, dW0 + st * kSt16 + kk * 128, kIdSt,
                   !(inf.first && kk == 0));
        mma_commit(&bars[kEmpty0 + st]);
        if (inf.last) mma_commit(&bars[kAccFull0 + ab]);
      }
      __syncwarp();
      issued = true;
      if (inf.last) ++uc;
      ++it;
    }
  mma_done:
#undef MMA_WAIT
    if (lane == 0) {
      if (issued) mma_commit(&bars[kMmaDone]);
      else mbar_arrive(&bars[kMmaDone]);
      if (!wait_bar(&bars[kMmaDone], 0, wns)) fail(SSD_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ math warps
    const int q = warp & 3, cq = warp >> 2;
    const int r = 32 * q + lane;  // tensor-memory lane: state row n
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint32_t it = 0, uc = 0;
    float later = 0.f;  // log2-decay of the unit's chunks already walked (later in time)
    bool pending = false;
    int pu = 0, pab = 0;
    uint32_t ppar = 0;
    float plater = 0.f;
    auto arrive = [&](int bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bar]);
    };
    // H_loc of a finished unit: lane n, columns p = 16 cq .. of both halves
    auto readout = [&]() -> bool {
      if (!wait_bar_warp(&bars[kAccFull0 + pab], ppar, wns)) return false;
      tc_fence_after();
      const uint32_t base = tmem + pab * 128 + lane_addr + 16 * cq;
      float a[16], b[16];
      tmem_ld16(base, a);
      tmem_ld16(base + 64, b);
      tmem_ld_wait();
      tie16(a);
      tie16(b);
      tc_fence_before();
      arrive(kAccFree0 + pab);
      float* dst = prm.slots + (long long)pu * kPN + (16 * cq) * kN + r;
#pragma unroll
      for (int k = 0; k < 16; ++k) __stcg(dst + k * kN, a[k] + b[k]);
      if (tid == 0) prm.dec[pu] = plater;
      return true;
    };
#define MATH_TRY(expr)     \
  if (!(expr)) {           \
    fail(SSD_ERR_TIMEOUT); \
    goto math_done;        \
  }
    while (true) {
      const int st = (int)(it % kStages);
      MATH_TRY(wait_bar_warp(&bars[kFull0 + st], (it / kStages) & 1u, wns));
      const TileInfo inf = *info(st);
      if (inf.kind == kKindEnd || __any_sync(0xffffffffu, *abort_v)) break;
      if (inf.first) later = 0.f;
      const float c2l = c2(st)[kQ - 1];
      const float wl = later + c2l;
      // w o X hi over the x tile in place (each item is read, then rewritten,
      // by the same thread), lo into the next tile
      wx_item(X(st), c2(st), dtt(st), tid, wl, X(st));
      wx_item(X(st), c2(st), dtt(st), tid + 512, wl, X(st));
      fence_proxy_async_smem();
      arrive(kWxFull0 + st);
      later += c2l;
      if (pending) {
        MATH_TRY(readout());
        pending = false;
      }
      if (inf.last) {
        pending = true;
        pu = inf.unit;
        plater = later;
        pab = uc & 1;
        ppar = (uc >> 1) & 1u;
        ++uc;
      }
      ++it;
    }
    if (pending) MATH_TRY(readout());
  math_done:;
#undef MATH_TRY
  }
#undef fail
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp) tmem_dealloc(tmem, kTmemCols);
}
}  // namespace k1

// ============================================================== kernel 2
// One thread per float4 of a (sequence, head) state; walks the segments.
__global__ void __launch_bounds__(256)
    ssd_seg_pass_kernel(const int32_t* uoff, int nseq, int H, float* slots, const float* dec,
                        const float* init, float* final_states) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kV = kPN / 4;  // float4 per state
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long sh = gid / kV;
  const int e4 = (int)(gid % kV);
  if (sh >= (long long)nseq * H) return;
  if (uoff[nseq + 1] != 0) return;
  const int s = (int)(sh / H), h = (int)(sh % H);
  const int u0 = uoff[s];
  const int ns = (uoff[s + 1] - u0) / H;
  if (ns == 0) return;  // no tokens: the plan kernel wrote final = init
  float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (init) hv = __ldg(reinterpret_cast<const float4*>(init + sh * kPN) + e4);
  float4* base = reinterpret_cast<float4*>(slots) + e4;
  for (int s0 = 0; s0 < ns; s0 += 8) {
    // the segments' local states are independent loads: issue eight at once
    float4 v[8];
    float d[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (s0 + k < ns) {
        const long long u = u0 + (long long)(s0 + k) * H + h;
        v[k] = __ldcg(base + u * kV);
        d[k] = fast_exp2(__ldcg(dec + u));
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (s0 + k < ns) {
        const long long u = u0 + (long long)(s0 + k) * H + h;
        __stcg(base + u * kV, hv);  // the state entering segment s0 + k
        hv.x = fmaf(d[k], hv.x, v[k].x);
        hv.y = fmaf(d[k], hv.y, v[k].y);
        hv.z = fmaf(d[k], hv.z, v[k].z);
        hv.w = fmaf(d[k], hv.w, v[k].w);
      }
    }
  }
  if (final_states) reinterpret_cast<float4*>(final_states + sh * kPN)[e4] = hv;
}

// ============================================================== kernel 3
namespace k3 {
// Warps 0-7: decay masks and the epilogue (two per tensor-memory lane
// quarter); 8-15: the running state (two per lane quarter, 32 of the 64
// headdim columns each); 16: producer; 17: MMA issuer.
constexpr int kMaskWarps = 8;
constexpr int kStateWarps = 8;
constexpr int kProducerWarp3 = 16;
constexpr int kMmaWarp3 = 17;
constexpr int kThreads3 = 576;
constexpr uint32_t kCBBytes = 4 * kTile;              // C (2 halves), B (2 halves)
constexpr uint32_t kOffX = 2 * kCBBytes;              // 2 x slots
constexpr uint32_t kOffW = kOffX + 2 * kTile;         // w o X hi, lo
constexpr uint32_t kOffHt = kOffW + 2 * kTile;        // H^T hi, lo
constexpr uint32_t kOffTabs = kOffHt + 2 * kTile;     // per x slot: the chunk's decay tables
constexpr uint32_t kOffInfo = kOffTabs + 2 * kTabBytes;
constexpr uint32_t kOffBars = kOffInfo + 2 * 64;
constexpr uint32_t kBarBytes = 24 * 8;
constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 16;
static_assert(kSmemBytes <= 232448, "shared memory per block");
// Tensor memory: two G / S' buffers, the forward accumulator
// [C H_hi^T + S' X | C H_lo^T] (lane i, column p of each half) and the
// chunk-state product [B^T (w o X)_hi | _lo] (lane n, column p of each half).
constexpr uint32_t kColG = 0;
constexpr uint32_t kColAcc = 256;
constexpr uint32_t kColSt = 384;
constexpr uint32_t kTmemCols = 512;

enum {
  kCbFull0 = 0, kCbFull1,      // C/B slot loaded (TMA)
  kCbEmpty0 = 2, kCbEmpty1,    // C/B slot read (MMA commit)
  kXFull0 = 4, kXFull1,        // x slot loaded (TMA) and its tables written
  kXEmpty0 = 6, kXEmpty1,      // x slot read (math warps + MMA commit)
  kGFull0 = 8, kGFull1,        // C B^T in G buffer (MMA commit)
  kSFull = 10,                 // S' written (mask warps)
  kHtFull = 11, kHtFree = 12,  // H^T operand tiles
  kAccFull = 13, kAccFree = 14,
  kWxFull = 15,                // w o X written (state warps; also: the previous
                               // chunk state has been read)
  kStFull = 16,                // chunk-state product
  kMmaDone = 17,
  kNumBars
};
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");

struct Params {
  UnitPlan up;
  const uint8_t* tabs;  // per (global chunk, head): decay tables
  const float* D;
  const float* hin;  // per unit: the state entering the segment [P][N] fp32
  float* y;
  int* ticket;       // ticket[1]: line of the first expired wait; ticket[2]: work ticket
  int32_t* status;
  int y_v8;          // y is 32-byte aligned: 32-byte stores
  unsigned long long wait_ns;
  int hold_unit;     // test hook: this unit's first mask is never published (-1: none)
};

__global__ void __launch_bounds__(kThreads3, 1)
    ssd_seg_out_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_c, Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (tid == 0) report(prm.status, SSD_ERR_UNSUPPORTED);
    return;
  }
  uint8_t* const sb = smem_raw;
  auto Cs = [&](int cb) { return sb + cb * kCBBytes; };
  auto Bs = [&](int cb) { return sb + cb * kCBBytes + 2 * kTile; };
  auto Xs = [&](int xs) { return sb + kOffX + xs * kTile; };
  uint8_t* const Wt = sb + kOffW;
  uint8_t* const Ht = sb + kOffHt;
  auto c2 = [&](int xs) { return reinterpret_cast<float*>(sb + kOffTabs + xs * kTabBytes); };
  auto Et = [&](int xs) {
    return reinterpret_cast<float*>(sb + kOffTabs + xs * kTabBytes + 512);
  };
  auto dtt = [&](int xs) {
    return reinterpret_cast<__nv_bfloat16*>(sb + kOffTabs + xs * kTabBytes + 1024);
  };
  auto info = [&](int xs) { return reinterpret_cast<TileInfo*>(sb + kOffInfo) + xs; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kOffBars);
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(sb + kOffBars + kBarBytes);
  int* abort_p = reinterpret_cast<int*>(sb + kOffBars + kBarBytes + 4);
  const unsigned long long wns = prm.wait_ns;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kCbFull0 + b], 1);
      mbar_init(&bars[kCbEmpty0 + b], 1);
      mbar_init(&bars[kXFull0 + b], 1);               // expect-tx arrival (tile, tables)
      mbar_init(&bars[kXEmpty0 + b], kMaskWarps + kStateWarps + 1);  // math warps + MMA
      mbar_init(&bars[kGFull0 + b], 1);
    }
    mbar_init(&bars[kSFull], kMaskWarps);
    mbar_init(&bars[kHtFull], kStateWarps);
    mbar_init(&bars[kHtFree], 1);
    mbar_init(&bars[kAccFull], 1);
    mbar_init(&bars[kAccFree], kMaskWarps);
    mbar_init(&bars[kWxFull], kStateWarps);
    mbar_init(&bars[kStFull], 1);
    mbar_init(&bars[kMmaDone], 1);
    *abort_p = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp3) {
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

  // the entering states (state-passing kernel) are ready past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nseq = prm.up.si.nseq;
  const int nunits = prm.up.uoff[nseq];
  const bool plan_ok = prm.up.uoff[nseq + 1] == 0;

  if (warp == kProducerWarp3) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map_x);
      prefetch_tmap(&map_b);
      prefetch_tmap(&map_c);
    }
    auto draw = [&](Unit& Xu) -> bool {
      int v = 0;
      if (lane == 0) v = atomicAdd(prm.ticket + 2, 1);
      v = __shfl_sync(0xffffffffu, v, 0);
      if (v >= nunits) return false;
      prm.up.decode(v, Xu);
      Xu.D = prm.D ? prm.D[Xu.h] : 0.f;
      return true;
    };
    uint32_t it = 0;
    bool ok = true, cb_only = false;
    Unit U, V;
    bool have = plan_ok && draw(U);
    int k = 0;
    auto coords = [&](const Unit& Xu, int kk, long long& t0, int& len) {
      t0 = Xu.b + (long long)(Xu.tb + kk) * kQ;
      len = (int)min((long long)kQ, Xu.e - t0);
    };
    if (have && lane == 0) bulk_prefetch_l2(prm.hin + (long long)U.u * kPN, kPN * 4);
    while (have) {
      const Unit Cu = U;
      const int kc = k;
      long long t0;
      int len;
      coords(Cu, kc, t0, len);
      const bool last = kc == Cu.n - 1;
      // the next unit is taken when its predecessor's last chunk is loaded
      bool have_next = false;
      if (last) {
        have_next = draw(V);
        // the state entering the next unit into L2 for the state warps
        if (have_next && lane == 0) bulk_prefetch_l2(prm.hin + (long long)V.u * kPN, kPN * 4);
        have = have_next;
        if (have) U = V;
        k = 0;
      } else {
        ++k;
      }
      const int s = it & 1;
      const uint32_t pe = ((it >> 1) - 1) & 1u;
      // C and B tiles (freed once the chunk's C H^T has run)
      if (it >= 2 && !wait_bar_warp(&bars[kCbEmpty0 + s], pe, wns)) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, *abort_v)) { ok = false; break; }
      if (lane == 0) {
        uint64_t* fcb = &bars[kCbFull0 + s];
        mbar_arrive_expect_tx(fcb, 4 * kTile);
        tma_load_2d(Bs(s), &map_b, fcb, Cu.g * kN, (int)t0);
        tma_load_2d(Bs(s) + kTile, &map_b, fcb, Cu.g * kN + 64, (int)t0);
        tma_load_2d(Cs(s), &map_c, fcb, Cu.g * kN, (int)t0);
        tma_load_2d(Cs(s) + kTile, &map_c, fcb, Cu.g * kN + 64, (int)t0);
      }
      // x tile and tables (freed once S' X and the math warps are done with them)
      if (it >= 2 && !wait_bar_warp(&bars[kXEmpty0 + s], pe, wns)) {
        if (lane == 0) fail(SSD_ERR_TIMEOUT);
        ok = false;
        cb_only = true;  // this chunk's C/B loads are in flight
        break;
      }
      if (lane == 0) {
        uint64_t* fx = &bars[kXFull0 + s];
        TileInfo* inf = info(s);
        inf->t0 = t0;
        inf->unit = Cu.u;
        inf->h = Cu.h;
        inf->len = len;
        inf->kind = kKindChunk;
        inf->first = kc == 0;
        inf->last = last;
        inf->next_unit = (last && have_next) ? V.u : -1;
        inf->D = Cu.D;
        const int gc = Cu.c0 + Cu.tb + kc;
        mbar_arrive_expect_tx(fx, kTile + kTabBytes);
        tma_load_2d(Xs(s), &map_x, fx, Cu.h * kP, (int)t0);
        bulk_load(c2(s), prm.tabs + ((long long)gc * prm.up.H + Cu.h) * kTabBytes, kTabBytes, fx);
        // the next chunk's x into L2 behind this one
        if (have) {
          long long nt0;
          int nlen;
          coords(U, k, nt0, nlen);
          tma_prefetch_2d(&map_x, U.h * kP, (int)nt0);
        }
      }
      __syncwarp();
      ++it;
    }
    const int s = it & 1;
    if (ok && (it < 2 || wait_bar_warp(&bars[kXEmpty0 + s], ((it >> 1) - 1) & 1u, wns))) {
      if (lane == 0) {
        info(s)->kind = kKindEnd;
        mbar_arrive(&bars[kXFull0 + s]);
      }
    } else if (lane == 0) {
      if (ok) fail(SSD_ERR_TIMEOUT);
      // aborting: loads still in flight must land before the CTA may exit
      for (uint32_t q = (it >= 2 ? it - 2 : 0); q < it; ++q) {
        (void)wait_bar(&bars[kCbFull0 + (q & 1)], (q >> 1) & 1u, wns);
        (void)wait_bar(&bars[kXFull0 + (q & 1)], (q >> 1) & 1u, wns);
      }
      if (cb_only) (void)wait_bar(&bars[kCbFull0 + s], (it >> 1) & 1u, wns);
    }
  } else if (warp == kMmaWarp3) {
    // ------------------------------------------------------------ MMA issuer
    // Per chunk t: S_t (unless t ends its unit), C H_t^T, S'_t X_t, then the
    // next chunk's C B^T into the other G buffer.
    const uint64_t dC0 = sdesc_sw128(smem_u32(Cs(0)), 16, 1024);      // K-major C
    const uint64_t dB0 = sdesc_sw128(smem_u32(Bs(0)), 16, 1024);      // K-major B
    const uint64_t dBt0 = sdesc_sw128(smem_u32(Bs(0)), kTile, 1024);  // MN-major B^T
    const uint64_t dW = sdesc_sw128(smem_u32(Wt), kTile, 1024);       // [w o X hi | lo]
    const uint64_t dX0 = sdesc_sw128(smem_u32(Xs(0)), kTile, 1024);   // MN-major x
    const uint64_t dHt = sdesc_sw128(smem_u32(Ht), kTile, 1024);      // [H hi | lo]^T
    constexpr uint64_t kCB16 = kCBBytes >> 4;
    uint32_t su = 0;
    bool issued = false;
    bool cur_last = false;
#define MMA_WAIT(bar, par)                      \
  if (!wait_bar_warp(&bars[bar], (par), wns)) { \
    if (lane == 0) fail(SSD_ERR_TIMEOUT);       \
    goto mma_done;                              \
  }
    MMA_WAIT(kXFull0, 0);
    if (info(0)->kind == kKindEnd || *abort_v) goto mma_done;
    cur_last = info(0)->last;
    MMA_WAIT(kCbFull0, 0);
    tc_fence_after();
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + kColG, dC0 + (kk >> 2) * kT16 + (kk & 3) * 2,
                 dB0 + (kk >> 2) * kT16 + (kk & 3) * 2, kIdG, kk > 0);
      mma_commit(&bars[kGFull0]);
    }
    __syncwarp();
    issued = true;
    for (uint32_t t = 0;; ++t) {
      const int s = t & 1;
      if (!cur_last) {
        // (w o X of this chunk is written after the previous chunk state was read)
        MMA_WAIT(kWxFull, su & 1u);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem + kColSt, dBt0 + s * kCB16 + kk * 128, dW + kk * 128, kIdSt, kk > 0);
          mma_commit(&bars[kStFull]);
        }
        __syncwarp();
        ++su;
      }
      MMA_WAIT(kHtFull, t & 1u);
      if (t > 0) { MMA_WAIT(kAccFree, (t - 1) & 1u); }
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tmem + kColAcc, dC0 + s * kCB16 + (kk >> 2) * kT16 + (kk & 3) * 2,
                   dHt + kk * 128, kIdCH, kk > 0);
        mma_commit(&bars[kHtFree]);
        mma_commit(&bars[kCbEmpty0 + s]);
      }
      __syncwarp();
      // the next chunk's C B^T, ahead of this chunk's S' X (the other G buffer)
      const int n = s ^ 1;
      MMA_WAIT(kXFull0 + n, ((t + 1) >> 1) & 1u);
      const bool more = !(info(n)->kind == kKindEnd || *abort_v);
      const bool next_last = more && info(n)->last;
      if (more) {
        // (G buffer n was last read by S' X of chunk t - 1, complete since the
        // epilogue warps released its accumulator before C H_t^T)
        MMA_WAIT(kCbFull0 + n, ((t + 1) >> 1) & 1u);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem + kColG + n * 128, dC0 + n * kCB16 + (kk >> 2) * kT16 + (kk & 3) * 2,
                     dB0 + n * kCB16 + (kk >> 2) * kT16 + (kk & 3) * 2, kIdG, kk > 0);
          mma_commit(&bars[kGFull0 + n]);
        }
        __syncwarp();
      }
      MMA_WAIT(kSFull, t & 1u);
      tc_fence_after();
      if (elect_one()) {
        const uint32_t scol = tmem + kColG + s * 128;
        // S' K block kk (columns j = 16 kk ..): 8 columns of hi pairs, then 8 of lo
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_tmem_a(tmem + kColAcc, scol + 16 * kk + 8 * part, dX0 + s * kT16 + kk * 128,
                            kIdSX, true);
        mma_commit(&bars[kAccFull]);
        mma_commit(&bars[kXEmpty0 + s]);
      }
      __syncwarp();
      if (!more) break;
      cur_last = next_last;
    }
  mma_done:
#undef MMA_WAIT
    if (lane == 0) {
      if (issued) mma_commit(&bars[kMmaDone]);
      else mbar_arrive(&bars[kMmaDone]);
      if (!wait_bar(&bars[kMmaDone], 0, wns)) fail(SSD_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ math warps
    // Three groups, each walking the chunks with its own barriers; warp w
    // reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31 only.
    const int q = warp & 3;
    const int r = 32 * q + lane;  // tensor-memory lane: token row i / state row n
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    auto arrive = [&](int bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bar]);
    };
#define MATH_TRY(expr)     \
  if (!(expr)) {           \
    fail(SSD_ERR_TIMEOUT); \
    goto math_done;        \
  }
    if (warp < kMaskWarps) {
      // ---------------- mask and epilogue warps.  Iteration t: y of chunk
      // t - 1 (its accumulator is complete once S'_{t-1} X has run), then
      // the mask S' of chunk t over its C B^T in place.  Warp w takes the
      // 32 x 32 blocks (rows 32 q.., columns 32 cq..) for cq = 2 hf, 2 hf + 1
      // (hf = w / 4), each in two 16-column halves rewritten as one K block:
      // 8 columns of hi pairs, then 8 of lo pairs; blocks above the diagonal
      // become zeros.  Its share of y is row r, columns p = 32 hf ...
      const int hf = warp >> 2;
      long long pt0 = 0;  // the previous chunk: first token, rows, head, row factor
      int plen = 0, ph = 0;
      float pf = 0.f;
      for (uint32_t t = 0;; ++t) {
        const int xs = t & 1;
        MATH_TRY(wait_bar_warp(&bars[kXFull0 + xs], (t >> 1) & 1u, wns));
        const TileInfo inf = *info(xs);
        const bool end = inf.kind == kKindEnd || __any_sync(0xffffffffu, *abort_v);
        if (t > 0) {
          // y = f (S' X + C H^T) of chunk t - 1
          MATH_TRY(wait_bar_warp(&bars[kAccFull], (t - 1) & 1u, wns));
          tc_fence_after();
          const uint32_t base = tmem + kColAcc + lane_addr + 32 * hf;
          float* yp = prm.y + ((pt0 + r) * prm.up.H + ph) * kP + 32 * hf;
          const bool row_ok = r < plen;
#pragma unroll
          for (int c0 = 0; c0 < 32; c0 += 16) {
            float a[16], b[16];
            tmem_ld16(base + c0, a);
            tmem_ld16(base + 64 + c0, b);
            tmem_ld_wait();
            tie16(a);
            tie16(b);
            if (c0 == 16) {
              tc_fence_before();
              arrive(kAccFree);
            }
            float o[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const f2 v = mul2(add2(f2{a[2 * k], a[2 * k + 1]}, f2{b[2 * k], b[2 * k + 1]}),
                                f2{pf, pf});
              o[2 * k] = v.x;
              o[2 * k + 1] = v.y;
            }
            if (row_ok) {
              if (prm.y_v8) {
                st_global_cs_v8(yp + c0, o);
                st_global_cs_v8(yp + c0 + 8, o + 8);
              } else {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                  __stcs(reinterpret_cast<float4*>(yp + c0) + m,
                         make_float4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]));
              }
            }
          }
        }
        if (end) break;
        MATH_TRY(wait_bar_warp(&bars[kGFull0 + xs], (t >> 1) & 1u, wns));
        tc_fence_after();
        const float c2r = c2(xs)[r];
        const float Dh = inf.D;
        const bool fast = __all_sync(0xffffffffu, c2r >= kDeep);
        const float mr = fmaxf(c2r, kDeep);
        const float Dr = Dh * fast_exp2(-mr);
        const float dr = c2r - mr;
#pragma unroll 1
        for (int bi = 0; bi < 2; ++bi) {
          const int cq = 2 * hf + bi;
          const uint32_t scol = tmem + kColG + xs * 128 + lane_addr + 32 * cq;
          if (cq > q) {
            uint32_t z[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) z[m] = 0u;
            tmem_st16(scol, z);
            tmem_st16(scol + 16, z);
            continue;
          }
          const bool diag = cq == q;
          float gg[2][16];
          tmem_ld16(scol, gg[0]);
          tmem_ld16(scol + 16, gg[1]);
          tmem_ld_wait();
          tie16(gg[0]);
          tie16(gg[1]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int j0 = 32 * cq + 16 * half;
            const float (&g)[16] = gg[half];
            f2 v[8];
            if (fast) {
              // every row's factor is exp(cum_i): S' = G E_j
              const float4* E4 = reinterpret_cast<const float4*>(Et(xs) + j0);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const float4 e = E4[m];
                v[2 * m] = mul2(f2{g[4 * m], g[4 * m + 1]}, f2{e.x, e.y});
                v[2 * m + 1] = mul2(f2{g[4 * m + 2], g[4 * m + 3]}, f2{e.z, e.w});
              }
            } else {
              // some rows decayed below 2^-60: exp2(c2_i - m_i - c2_j) dt_j per entry
              const float4* c4 = reinterpret_cast<const float4*>(c2(xs) + j0);
              const uint2* d2 = reinterpret_cast<const uint2*>(dtt(xs) + j0);
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
        if (!(inf.first && inf.unit == prm.hold_unit)) arrive(kSFull);
        pt0 = inf.t0;
        plen = inf.len;
        ph = inf.h;
        pf = fast_exp2(mr);
        arrive(kXEmpty0 + xs);
      }
    } else {
      // ---------------- state warps: the running state H[p][n = r] (fp32,
      // p = 32 hp .. 32 hp + 31 in registers, hp = (w - 8) / 4), its part of
      // the H^T operand and of w o X of the next chunk (row j = r).
      const int hp = (warp - kMaskWarps) >> 2;
      constexpr int kPh = kP / 2;
      float hs[kPh];
      auto load_state = [&](int unit) {
        const float* src = prm.hin + (long long)unit * kPN + (kPh * hp) * kN + r;
#pragma unroll
        for (int p = 0; p < kPh; ++p) hs[p] = __ldcg(src + p * kN);
      };
      // H^T (hi, lo) as the B operand of C H^T: row n = r, chunks 4 hp .. 4 hp + 3
      auto put_ht = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 h4, l4;
          split2p(f2{hs[8 * c + 0], hs[8 * c + 1]}, h4.x, l4.x);
          split2p(f2{hs[8 * c + 2], hs[8 * c + 3]}, h4.y, l4.y);
          split2p(f2{hs[8 * c + 4], hs[8 * c + 5]}, h4.z, l4.z);
          split2p(f2{hs[8 * c + 6], hs[8 * c + 7]}, h4.w, l4.w);
          const uint32_t off = sw128_offset(r, 4 * hp + c);
          *reinterpret_cast<uint4*>(Ht + off) = h4;
          *reinterpret_cast<uint4*>(Ht + kTile + off) = l4;
        }
        fence_proxy_async_smem();
        arrive(kHtFull);
      };
      // w o X of the chunk in x slot xs, row j = r, chunks 4 hp .. 4 hp + 3
      auto put_wx = [&](int xs) {
        const float w = fast_exp2(c2(xs)[kQ - 1] - c2(xs)[r]) * __bfloat162float(dtt(xs)[r]);
        const f2 ww{w, w};
        const uint8_t* xt = Xs(xs);
        uint4 xv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) xv[c] = *reinterpret_cast<const uint4*>(xt + sw128_offset(r, 4 * hp + c));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = sw128_offset(r, 4 * hp + c);
          uint4 hi, lo;
          split2p(mul2(bf2(xv[c].x), ww), hi.x, lo.x);
          split2p(mul2(bf2(xv[c].y), ww), hi.y, lo.y);
          split2p(mul2(bf2(xv[c].z), ww), hi.z, lo.z);
          split2p(mul2(bf2(xv[c].w), ww), hi.w, lo.w);
          *reinterpret_cast<uint4*>(Wt + off) = hi;
          *reinterpret_cast<uint4*>(Wt + kTile + off) = lo;
        }
        fence_proxy_async_smem();
        arrive(kWxFull);
      };
      uint32_t su = 0;
      MATH_TRY(wait_bar_warp(&bars[kXFull0], 0, wns));
      TileInfo cur = *info(0);
      if (cur.kind == kKindEnd || __any_sync(0xffffffffu, *abort_v)) goto math_done;
      load_state(cur.unit);
      if (!cur.last) put_wx(0);
      put_ht();
      float ca = fast_exp2(c2(0)[kQ - 1]);
      for (uint32_t t = 0;; ++t) {
        const int xs = t & 1, xn = xs ^ 1;
        MATH_TRY(wait_bar_warp(&bars[kXFull0 + xn], ((t + 1) >> 1) & 1u, wns));
        const TileInfo nx = *info(xn);
        const bool end = nx.kind == kKindEnd || __any_sync(0xffffffffu, *abort_v);
        if (!cur.last && !end) {
          // H_{t+1} = exp(cum_last) H_t + S_t
          MATH_TRY(wait_bar_warp(&bars[kStFull], su & 1u, wns));
          tc_fence_after();
          const uint32_t base = tmem + kColSt + lane_addr + kPh * hp;
#pragma unroll
          for (int c0 = 0; c0 < kPh; c0 += 16) {
            float a[16], b[16];
            tmem_ld16(base + c0, a);
            tmem_ld16(base + 64 + c0, b);
            tmem_ld_wait();
            tie16(a);
            tie16(b);
#pragma unroll
            for (int k2 = 0; k2 < 16; k2 += 2) {
              const f2 v = fma2(f2{ca, ca}, f2{hs[c0 + k2], hs[c0 + k2 + 1]},
                                add2(f2{a[k2], a[k2 + 1]}, f2{b[k2], b[k2 + 1]}));
              hs[c0 + k2] = v.x;
              hs[c0 + k2 + 1] = v.y;
            }
          }
          tc_fence_before();
          ++su;
        }
        arrive(kXEmpty0 + xs);
        if (end) break;
        if (nx.first) load_state(nx.unit);
        if (!nx.last) put_wx(xn);
        MATH_TRY(wait_bar_warp(&bars[kHtFree], t & 1u, wns));
        put_ht();
        ca = fast_exp2(c2(xn)[kQ - 1]);
        cur = nx;
      }
    }
  math_done:;
#undef MATH_TRY
  }
#undef fail
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarp3) tmem_dealloc(tmem, kTmemCols);
}
}  // namespace k3

struct WsLayout {
  size_t uoff, coff, ticket, tabs, slots, dec, total;
};

long long max_tc_chunks(const FwdArgs& a) {
  return max_chunks(a.batch, a.seqlen, kQ, a.cu != nullptr, a.nseq);
}

WsLayout ws_layout(const FwdArgs& a) {
  WsLayout L;
  const long long mu = tc_max_units(a);
  L.uoff = 0;
  L.coff = L.uoff + plan_bytes(a.nseq);
  L.ticket = L.coff + plan_bytes(a.nseq);
  L.tabs = L.ticket + 256;
  L.slots = L.tabs + align256((size_t)max_tc_chunks(a) * a.H * kTabBytes);
  L.dec = L.slots + align256(sizeof(float) * (size_t)mu * kPN);
  L.total = L.dec + align256(sizeof(float) * (size_t)mu);
  return L;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

bool tc3_supported(const FwdArgs& a) {
  return a.dtype == SSD_DT_BF16 && a.P == kP && a.N == kN && !a.dt_softplus && !a.z &&
         !a.y_bf16;
}

size_t tc3_workspace_bytes(const FwdArgs& a) { return ws_layout(a).total; }

namespace {

// Plan, decay tables, segment states and state passing: everything of the
// forward but the outputs.  Fills `p3` (when given) for the output kernel.
ssd_status_t states_pass(const FwdArgs& a, unsigned long long wait_ns, int hold_unit,
                         bool* work_out, CUtensorMap* mx, CUtensorMap* mb, k3::Params* p3,
                         int* grid_out) {
  const WsLayout L = ws_layout(a);
  char* ws = static_cast<char*>(a.ws);
  int32_t* uoff = reinterpret_cast<int32_t*>(ws + L.uoff);
  int32_t* coff = reinterpret_cast<int32_t*>(ws + L.coff);
  int* ticket = reinterpret_cast<int*>(ws + L.ticket);
  uint8_t* tabs = reinterpret_cast<uint8_t*>(ws + L.tabs);
  float* slots = reinterpret_cast<float*>(ws + L.slots);
  float* dec = reinterpret_cast<float*>(ws + L.dec);
  const long long ntok = (long long)a.batch * a.seqlen;
  const long long mu = tc_max_units(a);
  const int seg = tc_choose_seg(a);
  const bool work = ntok > 0 && mu > 0;
  *work_out = work;
  if (work && (!tc_make_map_bf16(mx, a.x, ntok, (long long)a.H * kP) ||
               !tc_make_map_bf16(mb, a.B, ntok, (long long)a.G * kN)))
    return SSD_ERR_CUDA;
  UnitPlan up;
  up.uoff = uoff;
  up.coff = coff;
  up.si = SeqInfo{a.cu, a.seqlen, a.nseq};
  up.H = a.H;
  up.G = a.G;
  up.seg = seg;
  k1::Params p1;
  p1.up = up;
  p1.tabs = tabs;
  p1.slots = slots;
  p1.dec = dec;
  p1.ticket = ticket;
  p1.status = a.dev_status;
  p1.wait_ns = wait_ns;
  if (p3) {
    p3->up = up;
    p3->tabs = tabs;
    p3->D = a.D;
    p3->hin = slots;
    p3->y = a.y;
    p3->ticket = ticket;
    p3->status = a.dev_status;
    p3->y_v8 = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
    p3->wait_ns = wait_ns;
    p3->hold_unit = hold_unit;
  }
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k1::ssd_seg_state_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)k1::kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k3::ssd_seg_out_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)k3::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;
  if (tc_launch_plan(a, seg, uoff, ticket, nullptr, 0, coff) != cudaSuccess) return SSD_ERR_CUDA;
  if (!work) return SSD_OK;
  const int grid = (int)(mu < tc_sm_count() ? mu : tc_sm_count());
  *grid_out = grid;
  // Programmatic dependent launches: each kernel may start its set-up while
  // the previous one runs and waits for its results (griddepcontrol.wait).
  {
    const int32_t* cuoff = uoff;
    const int32_t* ccoff = coff;
    SeqInfo si{a.cu, a.seqlen, a.nseq};
    int H = a.H;
    const __nv_bfloat16* dtp = static_cast<const __nv_bfloat16*>(a.dt);
    const float* Ap = a.A;
    void* args[] = {&cuoff, &ccoff, &si, &H, &dtp, &Ap, &tabs};
    const dim3 blocks((unsigned)max_tc_chunks(a), (unsigned)((a.H + kTabHeads - 1) / kTabHeads));
    if (launch_pdl(reinterpret_cast<const void*>(ssd_chunk_tables_kernel), blocks, dim3(256),
                   0, a.stream, args) != cudaSuccess)
      return SSD_ERR_CUDA;
  }
  {
    void* args[] = {mx, mb, &p1};
    if (launch_pdl(reinterpret_cast<const void*>(k1::ssd_seg_state_kernel), dim3(grid),
                   dim3(kThreads), k1::kSmemBytes, a.stream, args) != cudaSuccess)
      return SSD_ERR_CUDA;
  }
  {
    const int32_t* cuoff = uoff;
    int nseq = a.nseq, H = a.H;
    const float* init = a.init;
    float* fin = a.final_states;
    void* args[] = {&cuoff, &nseq, &H, &slots, &dec, &init, &fin};
    const long long threads = (long long)a.nseq * a.H * (kPN / 4);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (launch_pdl(reinterpret_cast<const void*>(ssd_seg_pass_kernel), dim3(blocks), dim3(256),
                   0, a.stream, args) != cudaSuccess)
      return SSD_ERR_CUDA;
  }
  count_launches(3);
  return SSD_OK;
}

}  // namespace

ssd_status_t tc3_states(const FwdArgs& a, unsigned long long wait_ns) {
  bool work = false;
  int grid = 0;
  CUtensorMap mx, mb;
  const ssd_status_t st = states_pass(a, wait_ns, -1, &work, &mx, &mb, nullptr, &grid);
  if (st != SSD_OK) return st;
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t tc3_forward(const FwdArgs& a, unsigned long long wait_ns, int hold_unit) {
  bool work = false;
  int grid = 0;
  CUtensorMap mx, mb, mc;
  k3::Params p3;
  const long long ntok = (long long)a.batch * a.seqlen;
  if (ntok > 0 && !tc_make_map_bf16(&mc, a.C, ntok, (long long)a.G * kN)) return SSD_ERR_CUDA;
  ssd_status_t st = states_pass(a, wait_ns, hold_unit, &work, &mx, &mb, &p3, &grid);
  if (st != SSD_OK || !work) return st;
  void* args[] = {&mx, &mb, &mc, &p3};
  if (launch_pdl(reinterpret_cast<const void*>(k3::ssd_seg_out_kernel), dim3(grid),
                 dim3(k3::kThreads3), k3::kSmemBytes, a.stream, args) != cudaSuccess)
    return SSD_ERR_CUDA;
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace ssd
