// ssd_tc_host.h -- host-side pieces shared by the tensor-core forward
// kernels (not part of the public ABI): TMA tensor maps, the plan kernel that
// lays out the work units, and the choice of segment length.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_internal.h"

namespace ssd {

// Tokens per chunk of the tensor-core kernels (the tcgen05 tile height M).
constexpr int kTcChunk = 128;
// Chunks per segment: dense batches take a length in [kTcSegMin, kTcSegMax]
// (see tc_choose_seg); packed sequences, whose lengths live on the device,
// take kTcSegVarlen.
constexpr int kTcSegMin = 4, kTcSegMax = 12, kTcSegVarlen = 8;

// SMs of the current device (queried once).
int tc_sm_count();

// Segment length for a call: dense batches pick, among kTcSegMin..kTcSegMax,
// the one whose units fill the SMs in the fewest chunk-steps (waves x chunks
// per unit), preferring longer segments on a tie.
int tc_choose_seg(const FwdArgs& a);

// Upper bound on the number of work units (sequence, segment, head) for any
// segment length a call may choose.
long long tc_max_units(const FwdArgs& a);

// 2-D bf16 map over a row-major [rows, cols] matrix, 64-column x 128-row
// boxes, 128-byte swizzle (the operand tiles of the MMAs).
bool tc_make_map_bf16(CUtensorMap* m, const void* ptr, long long rows, long long cols);
// y as a 2-D fp32 tensor [tokens][H * P]: 16-column x 32-row boxes, 64-byte
// swizzle (one math warp's staged tile).
bool tc_make_map_y_f32(CUtensorMap* m, float* ptr, long long rows, long long cols);
// fp32 [rows][cols]: 32-column (128-byte) x box_rows-row boxes, 128-byte
// swizzle (the backward's state tiles; box_rows <= 256).
bool tc_make_map_f32_sw128(CUtensorMap* m, float* ptr, long long rows, long long cols,
                           int box_rows);
// bf16 [rows][cols]: 32-column (64-byte) x box_rows-row boxes, 64-byte
// swizzle (the backward's state tiles as stored; box_rows <= 256).
bool tc_make_map_bf16_sw64(CUtensorMap* m, void* ptr, long long rows, long long cols,
                           int box_rows);
// bf16 [slabs][rows][cols] as a 3-D tensor: 64-column (128-byte) x 64-row x
// 1-slab boxes, 128-byte swizzle, zero fill past rows and cols (the
// backward's state tiles as loaded into the MMA operands).
bool tc_make_map_bf16_slab_sw128(CUtensorMap* m, const void* ptr, long long slabs, long long rows,
                                 long long cols);
// A 3-D tensor of bf16 (elem_bytes 2) or fp32 (4) values, dims d0 (innermost)
// .. d2, with b0 x b1 x b2 boxes, unswizzled or 128-byte swizzled; zero fill
// past the dims.
bool tc_make_map_3d(CUtensorMap* m, const void* ptr, int elem_bytes, long long d0, long long d1,
                    long long d2, int b0, int b1, int b2, bool sw128);
// bf16 y: 16-column (32-byte) x 32-row boxes, unswizzled.
bool tc_make_map_y_bf16(CUtensorMap* m, void* ptr, long long rows, long long cols);

// Plan kernel: per sequence the number of work units (segments of `seg`
// chunks x H heads) as offsets uoff[0..nseq], and uoff[nseq+1] = 0 if
// cu_seqlens is well formed (else SSD_ERR_INVALID in dev_status and no
// units); zeroes the work tickets (ticket[0..3]) and the first `max_units`
// hand-off flags; final = init (or 0) for sequences without tokens; when
// `coff` is given, the chunk offsets per sequence there (coff[0..nseq]).  It
// allows its dependent launch to start early (programmatic dependent launch).
cudaError_t tc_launch_plan(const FwdArgs& a, int seg, int32_t* uoff, int* ticket, int* flags,
                           long long max_units, int32_t* coff = nullptr);

}  // namespace ssd
