// ssd_tc_host.cu -- host-side pieces shared by the tensor-core forward
// kernels: TMA tensor maps, the plan kernel and the segment length choice.
#include <cuda.h>

#include <mutex>

#include "ssd_common.cuh"
#include "ssd_tc_host.h"

namespace ssd {
namespace {

// The plan kernel (see tc_launch_plan); one block of 1024 threads.
__global__ void __launch_bounds__(1024) tc_plan_kernel(const int32_t* cu, int seqlen_rows,
                                                       int seqlen_total, int nseq, int seg,
                                                       int H, int32_t* uoff, int* ticket,
                                                       int* flags, long long max_units,
                                                       const float* init, float* final_states,
                                                       int PN, int32_t* dev_status,
                                                       int32_t* coff) {
  // the forward kernel may be scheduled now; it waits for this grid's
  // completion before it reads anything written here
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ int buf[32];
  __shared__ int carry, bad;
  if (threadIdx.x == 0) {
    carry = 0;
    bad = 0;
    for (int k = 0; k < 4; ++k) ticket[k] = 0;
    if (cu && (cu[0] != 0 || cu[nseq] != seqlen_total)) bad = 1;
  }
  for (long long k = threadIdx.x; k < max_units; k += 1024) flags[k] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // pass 0: units per sequence into uoff; pass 1 (when coff is given):
  // chunks per sequence into coff
  for (int pass = 0; pass < (coff ? 2 : 1); ++pass) {
    int32_t* offs = pass == 0 ? uoff : coff;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < nseq; base += 1024) {
      const int s = base + threadIdx.x;
      int n = 0;
      if (s < nseq) {
        const long long b = cu ? (long long)cu[s] : (long long)s * seqlen_rows;
        const long long e = cu ? (long long)cu[s + 1] : (long long)(s + 1) * seqlen_rows;
        if (e < b || b < 0 || e > seqlen_total) atomicOr(&bad, 1);
        const long long nt = e > b ? (e - b + kTcChunk - 1) / kTcChunk : 0;
        n = pass == 0 ? (int)((nt + seg - 1) / seg) * H : (int)nt;
      }
      int v = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (lane == 31) buf[wid] = v;
      __syncthreads();
      int off = 0;
      for (int w = 0; w < wid; ++w) off += buf[w];
      if (s < nseq) offs[s + 1] = carry + v + off;
      __syncthreads();
      if (threadIdx.x == 1023) carry += v + off;
      __syncthreads();
    }
    if (threadIdx.x == 0) offs[0] = 0;
    __syncthreads();
  }
  if (bad) {
    for (int s = threadIdx.x; s <= nseq; s += 1024) {
      uoff[s] = 0;
      if (coff) coff[s] = 0;
    }
    if (threadIdx.x == 0) report(dev_status, SSD_ERR_INVALID);
  }
  if (threadIdx.x == 0) uoff[nseq + 1] = bad;
  __syncthreads();
  if (final_states && !bad) {
    const long long per = (long long)H * PN;
    for (int s = 0; s < nseq; ++s) {
      if (uoff[s + 1] != uoff[s]) continue;  // the sequence has tokens
      float* dst = final_states + (long long)s * per;
      const float* src = init ? init + (long long)s * per : nullptr;
      for (long long e = threadIdx.x; e < per; e += 1024) dst[e] = src ? src[e] : 0.f;
    }
  }
}

// --------------------------------------------------------------------------

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

}  // namespace

// 2-D bf16 map over a [rows, cols] row-major matrix, 64 x 128 boxes, 128B swizzle.
bool tc_make_map_bf16(CUtensorMap* m, const void* ptr, long long rows, long long cols) {
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

// y as a 2D fp32 tensor [tokens][H * P]; a box is 16 columns x 32 rows,
// 64B-swizzled (one math warp's tile).
bool tc_make_map_y_f32(CUtensorMap* m, float* ptr, long long rows, long long cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows][cols]: a box is 32 columns (128 bytes) x box_rows rows,
// 128-byte swizzle (the backward's state tiles).
bool tc_make_map_f32_sw128(CUtensorMap* m, float* ptr, long long rows, long long cols,
                           int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][cols] (the backward's hi/lo state tiles as the state scans
// store them): a box is 32 columns (64 bytes) x box_rows rows, 64-byte swizzle.
bool tc_make_map_bf16_sw64(CUtensorMap* m, void* ptr, long long rows, long long cols,
                           int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [slabs][rows][cols] (the same tiles as the gradient kernel loads
// them): a box is 64 columns (128 bytes) x 64 rows of one slab, 128-byte
// swizzle; elements past rows or cols read as zero.
bool tc_make_map_bf16_slab_sw128(CUtensorMap* m, const void* ptr, long long slabs, long long rows,
                                 long long cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)slabs};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(cols * rows) * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D bf16 or fp32 tensor (the backward scans' per-step operands: B or C
// rows of one group, x or dy rows of one head).
bool tc_make_map_3d(CUtensorMap* m, const void* ptr, int elem_bytes, long long d0, long long d1,
                    long long d2, int b0, int b1, int b2, bool sw128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)(d0 * elem_bytes), (cuuint64_t)(d0 * d1 * elem_bytes)};
  cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, (cuuint32_t)b2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 y (the fused-epilogue option): a box is 16 columns (32 bytes) x 32
// rows, unswizzled.
bool tc_make_map_y_bf16(CUtensorMap* m, void* ptr, long long rows, long long cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  });
  return n > 0 ? n : 148;
}

int tc_choose_seg(const FwdArgs& a) {
  if (a.cu) return kTcSegVarlen;
  const long long nt = ((long long)a.seqlen + kTcChunk - 1) / kTcChunk;
  const long long nsm = tc_sm_count();
  int best = kTcSegMax;
  long long best_cost = -1;
  for (int sg = kTcSegMax; sg >= kTcSegMin; --sg) {
    const long long units = (long long)a.batch * ((nt + sg - 1) / sg) * a.H;
    const long long cost = ((units + nsm - 1) / nsm) * (nt < sg ? nt : sg);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sg;
    }
  }
  return best;
}

long long tc_max_units(const FwdArgs& a) {
  const long long per = ((long long)a.seqlen + kTcChunk - 1) / kTcChunk;
  if (a.cu) return (((per + a.nseq) + kTcSegVarlen - 1) / kTcSegVarlen + a.nseq) * a.H;
  return (long long)a.batch * ((per + kTcSegMin - 1) / kTcSegMin) * a.H;
}

cudaError_t tc_launch_plan(const FwdArgs& a, int seg, int32_t* uoff, int* ticket, int* flags,
                           long long max_units, int32_t* coff) {
  const long long ntok = (long long)a.batch * a.seqlen;
  tc_plan_kernel<<<1, 1024, 0, a.stream>>>(a.cu, a.seqlen, (int)ntok, a.nseq, seg, a.H, uoff,
                                           ticket, flags, max_units, a.init, a.final_states,
                                           a.P * a.N, a.dev_status, coff);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace ssd
