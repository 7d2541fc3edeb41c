// ssd_simt.cu -- CUDA-core (SIMT, fp32 arithmetic) chunked SSD forward.
//
// This is the float32-input path (tensor-core operands cannot carry the
// 1e-4 relative accuracy that float32 inputs ask for) and the path for
// shapes the tcgen05 kernel does not cover.  It follows the four steps of
// the SSD chunked algorithm ("Transformers are SSMs Review", sec. 3-2 (4)),
// one kernel per step group:
//
//   simt_chunk_state  per (chunk, head): cumulative log-decay cum_i (sum of
//                     dt_k A over the chunk up to i), the chunk's decay
//                     exp(cum_last), and its state
//                     S_c[p,n] = sum_j exp(cum_last - cum_j) dt_j x_j[p] B_j[n]
//   simt_state_pass   per (sequence, head): H_c = exp(cum_last,c) H_{c-1} + S_c,
//                     H_{-1} = init; stores each chunk's input state H_{c-1}
//                     in place of S_c, and the final state
//   simt_chunk_out    per (chunk, head): y_i = sum_{j<=i} (C_i.B_j)
//                     exp(cum_i - cum_j) dt_j x_j + exp(cum_i) C_i H_{c-1}^T
//                     + D x_i
//
// Chunks never cross a sequence boundary (varlen packing cuts the state
// there, same review, sec. 3-2 (6)); the last chunk of a sequence may be
// short.
#include <cuda_bf16.h>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;  // token tile of the SIMT kernels

// Inclusive scan across a 256-thread block.  `buf` holds >= 8 floats.
__device__ __forceinline__ float block_scan_256(float v, float* buf) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) buf[wid] = v;
  __syncthreads();
  float off = 0.f;
  for (int w = 0; w < wid; ++w) off += buf[w];
  __syncthreads();
  return v + off;
}

__device__ __forceinline__ int block_scan_int_1024(int v, int* buf) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) buf[wid] = v;
  __syncthreads();
  int off = 0;
  for (int w = 0; w < wid; ++w) off += buf[w];
  __syncthreads();
  return v + off;
}

// Per-sequence chunk offsets.  One block of 1024 threads.  offs[nseq + 1]
// is the plan status: 0 = valid, else the cu_seqlens array was malformed
// and every offset is 0 (nothing is computed).  Optionally zeroes a work
// ticket and writes final = init (or 0) for sequences with no tokens.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* cu, int seqlen_rows,
                                                    int seqlen_total, int nseq, int q,
                                                    int32_t* offs, int32_t* dev_status,
                                                    int* ticket, const float* init,
                                                    float* final_states, int H, int PN) {
  if (ticket && threadIdx.x == 0) *ticket = 0;
  __shared__ int buf[32];
  __shared__ int carry, bad;
  if (threadIdx.x == 0) {
    carry = 0;
    bad = 0;
    if (cu && (cu[0] != 0 || cu[nseq] != seqlen_total)) bad = 1;
  }
  __syncthreads();
  for (int base = 0; base < nseq; base += 1024) {
    const int s = base + threadIdx.x;
    int n = 0;
    if (s < nseq) {
      long long b = cu ? (long long)cu[s] : (long long)s * seqlen_rows;
      long long e = cu ? (long long)cu[s + 1] : (long long)(s + 1) * seqlen_rows;
      if (e < b || b < 0 || e > seqlen_total) atomicOr(&bad, 1);
      n = e > b ? (int)((e - b + q - 1) / q) : 0;
    }
    const int incl = block_scan_int_1024(n, buf);
    if (s < nseq) offs[s + 1] = carry + incl;
    __syncthreads();
    if (threadIdx.x == 1023) carry += incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) offs[0] = 0;
  __syncthreads();
  if (bad) {
    for (int s = threadIdx.x; s <= nseq; s += 1024) offs[s] = 0;
    if (threadIdx.x == 0) report(dev_status, SSD_ERR_INVALID);
  }
  if (threadIdx.x == 0) offs[nseq + 1] = bad;
  if (final_states && !bad) {
    const long long per = (long long)H * PN;
    for (int s = 0; s < nseq; ++s) {
      if (offs[s + 1] != offs[s]) continue;  // sequence has tokens
      float* dst = final_states + (long long)s * per;
      const float* src = init ? init + (long long)s * per : nullptr;
      for (long long e = threadIdx.x; e < per; e += 1024) dst[e] = src ? src[e] : 0.f;
    }
  }
}

struct ChunkPos {
  int s;          // sequence
  long long t0;   // first token (flattened index)
  int len;        // tokens in this chunk (1..Q)
};

__device__ __forceinline__ bool locate(const int32_t* offs, const SeqInfo& si, int q, int g,
                                       ChunkPos& cp) {
  if (offs[si.nseq + 1] != 0) return false;  // malformed cu_seqlens
  if (g >= offs[si.nseq]) return false;
  cp.s = upper_index(offs, si.nseq, g);
  cp.t0 = si.begin(cp.s) + (long long)(g - offs[cp.s]) * q;
  cp.len = (int)min((long long)q, si.end(cp.s) - cp.t0);
  return true;
}

// cum[j] (j < len) = sum_{k<=j} dt_k * A_h, via a block scan; also stores dt.
template <typename Tin>
__device__ __forceinline__ void chunk_cumsum(const Tin* dt, const ChunkPos& cp, int H, int h,
                                             float Ah, int q, float* cum, float* dts,
                                             float* scanbuf) {
  for (int base = 0; base < q; base += kThreads) {
    const int j = base + threadIdx.x;
    float d = 0.f;
    if (j < cp.len) d = ld_in(dt + (cp.t0 + j) * H + h);
    float v = block_scan_256(d * Ah, scanbuf);
    if (base > 0) v += cum[base - 1];
    __syncthreads();
    if (j < q) {
      cum[j] = v;
      dts[j] = d;
    }
    __syncthreads();
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) simt_chunk_state(
    const Tin* __restrict__ x, const Tin* __restrict__ dt, const float* __restrict__ A,
    const Tin* __restrict__ B, SeqInfo si, const int32_t* __restrict__ offs, int H, int P, int N,
    int G, int q, float* __restrict__ states, float* __restrict__ decay) {
  ChunkPos cp;
  const int g = blockIdx.x, h = blockIdx.y;
  if (!locate(offs, si, q, g, cp)) return;
  const int grp = (int)((long long)h * G / H);
  extern __shared__ float sm[];
  float* cum = sm;              // [q]
  float* dts = cum + q;         // [q]
  float* xs = dts + q;          // [kTile][P], pre-scaled by the decay weight
  float* bs = xs + kTile * P;   // [kTile][N]
  __shared__ float scanbuf[8];
  chunk_cumsum(dt, cp, H, h, A[h], q, cum, dts, scanbuf);
  const float last = cum[cp.len - 1];
  // decay weight of token j in the chunk's final state, stored over dt
  for (int j = threadIdx.x; j < cp.len; j += kThreads) dts[j] = expf(last - cum[j]) * dts[j];
  __syncthreads();
  const int PN = P * N;
  constexpr int kMaxOut = 32;
  for (int o0 = 0; o0 < PN; o0 += kThreads * kMaxOut) {
    float acc[kMaxOut];
#pragma unroll
    for (int r = 0; r < kMaxOut; ++r) acc[r] = 0.f;
    for (int j0 = 0; j0 < cp.len; j0 += kTile) {
      const int nj = min(kTile, cp.len - j0);
      for (int e = threadIdx.x; e < kTile * P; e += kThreads) {
        const int jj = e / P, p = e % P;
        float v = 0.f;
        if (jj < nj) {
          const int j = j0 + jj;
          v = dts[j] * ld_in(x + ((cp.t0 + j) * H + h) * P + p);
        }
        xs[e] = v;
      }
      for (int e = threadIdx.x; e < kTile * N; e += kThreads) {
        const int jj = e / N, n = e % N;
        bs[e] = jj < nj ? ld_in(B + ((cp.t0 + j0 + jj) * G + grp) * N + n) : 0.f;
      }
      __syncthreads();
      for (int jj = 0; jj < nj; ++jj) {
#pragma unroll
        for (int r = 0; r < kMaxOut; ++r) {
          const int o = o0 + threadIdx.x + r * kThreads;
          if (o < PN) acc[r] += xs[jj * P + o / N] * bs[jj * N + o % N];
        }
      }
      __syncthreads();
    }
    float* dst = states + ((long long)g * H + h) * PN;
#pragma unroll
    for (int r = 0; r < kMaxOut; ++r) {
      const int o = o0 + threadIdx.x + r * kThreads;
      if (o < PN) dst[o] = acc[r];
    }
  }
  if (threadIdx.x == 0) decay[(long long)g * H + h] = expf(last);
}

// One block per (sequence, head, slice of the P*N state).  Sequential over
// the sequence's chunks: H_c = d_c H_{c-1} + S_c; S_c is replaced by H_{c-1}.
__global__ void __launch_bounds__(kThreads) simt_state_pass(
    const float* __restrict__ init, float* __restrict__ final_states, SeqInfo si,
    const int32_t* __restrict__ offs, int H, int PN, float* __restrict__ states,
    const float* __restrict__ decay) {
  if (offs[si.nseq + 1] != 0) return;
  const int s = blockIdx.x, h = blockIdx.y;
  const int e = (blockIdx.z * kThreads + threadIdx.x) * 4;
  if (e >= PN) return;
  float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
  if (init) cur = *reinterpret_cast<const float4*>(init + ((long long)s * H + h) * PN + e);
  for (int c = offs[s]; c < offs[s + 1]; ++c) {
    float4* slot = reinterpret_cast<float4*>(states + ((long long)c * H + h) * PN + e);
    const float4 sc = *slot;
    *slot = cur;
    const float d = decay[(long long)c * H + h];
    cur.x = d * cur.x + sc.x;
    cur.y = d * cur.y + sc.y;
    cur.z = d * cur.z + sc.z;
    cur.w = d * cur.w + sc.w;
  }
  if (final_states)
    *reinterpret_cast<float4*>(final_states + ((long long)s * H + h) * PN + e) = cur;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) simt_chunk_out(
    const Tin* __restrict__ x, const Tin* __restrict__ dt, const float* __restrict__ A,
    const Tin* __restrict__ B, const Tin* __restrict__ C, const float* __restrict__ D, SeqInfo si,
    const int32_t* __restrict__ offs, int H, int P, int N, int G, int q,
    const float* __restrict__ states, float* __restrict__ y) {
  ChunkPos cp;
  const int g = blockIdx.x, h = blockIdx.y;
  if (!locate(offs, si, q, g, cp)) return;
  const int grp = (int)((long long)h * G / H);
  const int NP = N + 1;  // padded row pitch of the C tile
  extern __shared__ float sm[];
  float* cum = sm;                 // [q]
  float* dts = cum + q;            // [q]
  float* cs = dts + q;             // [kTile][N+1]   C rows i
  float* bs = cs + kTile * NP;     // [kTile][N]     B rows j
  float* xs = bs + kTile * N;      // [kTile][P]     x rows j
  float* ws = xs + kTile * P;      // [kTile][kTile+1] masked weights
  float* hs = ws + kTile * (kTile + 1);  // [P][kTile] slice of H_{c-1}
  __shared__ float scanbuf[8];
  chunk_cumsum(dt, cp, H, h, A[h], q, cum, dts, scanbuf);
  const float Dh = D ? D[h] : 0.f;
  const float* Hprev = states + ((long long)g * H + h) * (long long)(P * N);
  const int r = threadIdx.x % kTile;  // row of the 32-row tile owned by this thread
  const int cg = threadIdx.x / kTile; // column group 0..7
  constexpr int kMaxP = 16;           // P <= 128 -> at most 16 columns per thread

  for (int i0 = 0; i0 < cp.len; i0 += kTile) {
    const int ni = min(kTile, cp.len - i0);
    float acc[kMaxP];
#pragma unroll
    for (int k = 0; k < kMaxP; ++k) acc[k] = 0.f;
    for (int e = threadIdx.x; e < kTile * N; e += kThreads) {
      const int ii = e / N, n = e % N;
      cs[ii * NP + n] = ii < ni ? ld_in(C + ((cp.t0 + i0 + ii) * G + grp) * N + n) : 0.f;
    }
    __syncthreads();
    // off-diagonal term: exp(cum_i) * sum_n C_i[n] H_{c-1}[p, n]
    for (int n0 = 0; n0 < N; n0 += kTile) {
      const int nlen = min(kTile, N - n0);  // N may be 16: a partial slice
      for (int e = threadIdx.x; e < P * kTile; e += kThreads) {
        const int p = e / kTile, nn = e % kTile;
        hs[e] = nn < nlen ? Hprev[(long long)p * N + n0 + nn] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxP; ++k) {
        const int p = cg + 8 * k;
        if (p < P) {
          float a = 0.f;
          for (int nn = 0; nn < nlen; ++nn) a += cs[r * NP + n0 + nn] * hs[p * kTile + nn];
          acc[k] += a;
        }
      }
      __syncthreads();
    }
    const float ecum = r < ni ? expf(cum[i0 + r]) : 0.f;
#pragma unroll
    for (int k = 0; k < kMaxP; ++k) acc[k] *= ecum;
    // diagonal block: sum over j <= i of (C_i.B_j) exp(cum_i - cum_j) dt_j x_j
    for (int j0 = 0; j0 <= i0 && j0 < cp.len; j0 += kTile) {
      const int nj = min(kTile, cp.len - j0);
      for (int e = threadIdx.x; e < kTile * N; e += kThreads) {
        const int jj = e / N, n = e % N;
        bs[e] = jj < nj ? ld_in(B + ((cp.t0 + j0 + jj) * G + grp) * N + n) : 0.f;
      }
      for (int e = threadIdx.x; e < kTile * P; e += kThreads) {
        const int jj = e / P, p = e % P;
        xs[e] = jj < nj ? ld_in(x + ((cp.t0 + j0 + jj) * H + h) * P + p) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int jj = cg + 8 * k;
        const int i = i0 + r, j = j0 + jj;
        float wv = 0.f;
        if (r < ni && jj < nj && j <= i) {
          float dot = 0.f;
          for (int n = 0; n < N; ++n) dot += cs[r * NP + n] * bs[jj * N + n];
          wv = dot * expf(cum[i] - cum[j]) * dts[j];
        }
        ws[r * (kTile + 1) + jj] = wv;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxP; ++k) {
        const int p = cg + 8 * k;
        if (p < P) {
          float a = 0.f;
          for (int jj = 0; jj < kTile; ++jj) a += ws[r * (kTile + 1) + jj] * xs[jj * P + p];
          acc[k] += a;
        }
      }
      __syncthreads();
    }
    if (r < ni) {
      const long long row = ((cp.t0 + i0 + r) * H + h) * (long long)P;
#pragma unroll
      for (int k = 0; k < kMaxP; ++k) {
        const int p = cg + 8 * k;
        if (p < P) y[row + p] = acc[k] + Dh * ld_in(x + row + p);
      }
    }
    __syncthreads();
  }
}

size_t out_smem(int q, int P, int N) {
  return sizeof(float) * (2 * q + kTile * (N + 1) + kTile * N + kTile * P + kTile * (kTile + 1) +
                          P * kTile);
}
size_t state_smem(int q, int P, int N) { return sizeof(float) * (2 * q + kTile * P + kTile * N); }

template <typename Tin>
ssd_status_t simt_forward_t(const FwdArgs& a) {
  const bool varlen = a.cu != nullptr;
  const long long mc = max_chunks(a.batch, a.seqlen, a.Q, varlen, a.nseq);
  char* ws = static_cast<char*>(a.ws);
  int32_t* offs = reinterpret_cast<int32_t*>(ws);
  ws += plan_bytes(a.nseq);
  float* decay = reinterpret_cast<float*>(ws);
  ws += align256(sizeof(float) * (size_t)mc * a.H);
  float* states = reinterpret_cast<float*>(ws);
  const long long total_tok = (long long)a.batch * a.seqlen;
  cudaError_t err = launch_plan(a.cu, a.seqlen, (int)total_tok, a.nseq, a.Q, offs, a.dev_status,
                                a.stream);
  if (err != cudaSuccess) return SSD_ERR_CUDA;
  SeqInfo si{a.cu, a.seqlen, a.nseq};
  const Tin* x = static_cast<const Tin*>(a.x);
  const Tin* dt = static_cast<const Tin*>(a.dt);
  const Tin* B = static_cast<const Tin*>(a.B);
  const Tin* C = static_cast<const Tin*>(a.C);
  const int PN = a.P * a.N;
  if (mc > 0) {
    const size_t sm1 = state_smem(a.Q, a.P, a.N);
    if (cudaFuncSetAttribute(simt_chunk_state<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm1) != cudaSuccess)
      return SSD_ERR_CUDA;
    simt_chunk_state<Tin><<<dim3((unsigned)mc, a.H), kThreads, sm1, a.stream>>>(
        x, dt, a.A, B, si, offs, a.H, a.P, a.N, a.G, a.Q, states, decay);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  if (a.nseq > 0) {
    dim3 grid(a.nseq, a.H, (PN / 4 + kThreads - 1) / kThreads);
    simt_state_pass<<<grid, kThreads, 0, a.stream>>>(a.init, a.final_states, si, offs, a.H, PN,
                                                      states, decay);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  if (mc > 0) {
    const size_t sm3 = out_smem(a.Q, a.P, a.N);
    if (cudaFuncSetAttribute(simt_chunk_out<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm3) != cudaSuccess)
      return SSD_ERR_CUDA;
    simt_chunk_out<Tin><<<dim3((unsigned)mc, a.H), kThreads, sm3, a.stream>>>(
        x, dt, a.A, B, C, a.D, si, offs, a.H, a.P, a.N, a.G, a.Q, states, a.y);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  }
  return SSD_OK;
}

}  // namespace

cudaError_t launch_plan(const int32_t* cu, int seqlen_rows, int seqlen_total, int nseq, int q,
                        int32_t* offs, int32_t* dev_status, cudaStream_t stream, int* ticket,
                        const float* init, float* final_states, int H, int PN) {
  plan_kernel<<<1, 1024, 0, stream>>>(cu, seqlen_rows, seqlen_total, nseq, q, offs, dev_status,
                                      ticket, init, final_states, H, PN);
  count_launches(1);
  return cudaGetLastError();
}

size_t simt_workspace_bytes(const FwdArgs& a) {
  const long long mc = max_chunks(a.batch, a.seqlen, a.Q, a.cu != nullptr, a.nseq);
  return plan_bytes(a.nseq) + align256(sizeof(float) * (size_t)mc * a.H) +
         align256(sizeof(float) * (size_t)mc * a.H * a.P * a.N);
}

ssd_status_t simt_forward(const FwdArgs& a) {
  return a.dtype == SSD_DT_BF16 ? simt_forward_t<__nv_bfloat16>(a) : simt_forward_t<float>(a);
}

}  // namespace ssd
