// sgemv_internal.cuh -- handle layout, device layout constants and launch
// declarations shared by the library's translation units.
//
// Device layout of a packed weight (all row-major over rows):
//   chunk  : 32 consecutive kept weights of one row = 16 "pair units" of two
//            kept weights each.  A row holds ceil(P / 32) chunks; a tail
//            chunk is zero-filled past the row's last kept weight, and the
//            row's chunk count in memory is rounded up to even (zero chunk)
//            so that every row of `idx` starts on a 16-byte boundary.
//   vals   : 16 bytes per chunk, identical to the canonical nibble order
//            (kept weight i of the chunk at bits 4*(i%8) of 32-bit word i/8).
//   idx    : 8 bytes per chunk, the canonical bits unchanged: pair unit u's
//            4-bit field a | b << 2 at bits 4*(u%8) of 32-bit word u/8.
//              N = 2: unit u is quad 16*chunk + u with ascending positions
//                     a < b (one of six fields);
//              N = 1: unit u is quads (32*chunk + 2u, 32*chunk + 2u + 1),
//                     a and b their positions.
//   sz     : 4 bytes per (row, group): binary16 scale in the low half,
//            binary16 zero in the high half; rows padded with zero words to
//            a multiple of 4 groups (16-byte aligned rows).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sgemv.h"

namespace sgemv {

constexpr int kChunkKept = 32;   // kept weights per chunk
constexpr int kUnitsPerChunk = 16;

struct Layout {
  int rows, cols, n_keep, group;
  int64_t kept;        // P, kept weights per row
  int64_t chunks;      // chunks holding the row's kept weights
  int64_t cstride;     // chunks per row in memory: `chunks` rounded up to even
  int64_t ngroups;     // cols / group
  int64_t gstride;     // scale/zero words per row in memory: multiple of 4
  int64_t vals_row;    // canonical bytes per row
  int64_t idx_row;
};

// Tensor maps of a packed weight for the tensor-core batch kernel, and its
// split-K workspace (fp32 partial tiles) and per-tile arrival counters.
struct TcMaps {
  CUtensorMap vals, idx, sz;
  float* scratch;
  int* counters;
  bool ready;
};

}  // namespace sgemv

struct sgemv_ctx {
  sgemv::Layout L;
  int max_m;
  int device;
  bool ready;
  uint4* d_vals;       // rows x chunks
  uint2* d_idx;        // rows x chunks
  uint32_t* d_sz;      // rows x ngroups
  __half* d_xstage;    // max_m x cols (sgemv_run_host)
  __half* d_ystage;    // max_m x rows
  int* d_err;          // device error word
  cudaStream_t stream; // private stream for pack / import / export
  // group size per row (NULL: every row uses L.group).  With per-row sizes
  // L.group is the finest of them and the device keeps scale/zero at that
  // granularity, a coarser group's words repeated in each of its sub-slots,
  // so the product kernels index groups uniformly.
  int* d_rowg;         // rows group sizes
  int64_t* d_goff;     // rows + 1 canonical scale/zero offsets
  int64_t canon_groups;  // canonical scale/zero entries of the whole matrix
  int withhold_runs;     // failure-detection test hook: runs left to sabotage
  sgemv::TcMaps tc;      // batch kernel (2 <= m): weight maps and split-K workspace
};

namespace sgemv {

// Error word values written by kernels (first error wins).
constexpr int kDevErrNonfinite = 1;
constexpr int kDevErrRange = 2;
constexpr int kDevErrBadIndex = 3;
constexpr int kDevErrTimeout = 4;
constexpr int kDevErrChecked = 5;   // checked build: a decoded code or index left its range

// The checked build (-DSGEMV_CHECKED, a debugging aid) makes the product
// kernels validate what they decode -- every 2:4 position nibble ascends,
// every group and chunk index stays inside its row -- and record
// kDevErrChecked instead of reading out of range (never a trap).
#ifdef SGEMV_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Nonzero unless each of the eight 2:4 position nibbles a | b << 2 of w has
// a < b.
__device__ __forceinline__ uint32_t bad_codes24(uint32_t w) {
  uint32_t bad = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t c = (w >> (4 * i)) & 0xFu;
    bad |= (uint32_t)((c & 3u) >= (c >> 2));
  }
  return bad;
}
__device__ __forceinline__ void report_checked(int* err) { atomicCAS(err, 0, kDevErrChecked); }

// ---- format kernels (sgemv_format.cu) ----
// Per-row group sizes of a matrix (rowg NULL: L.group for every row) and
// the canonical scale/zero offset of each row (goff NULL: r * L.ngroups).
struct RowGroups {
  const int* rowg;
  const int64_t* goff;
};

// xnorm (cols values) selects Eq. 3 importance pruning, with grad (rows x
// cols) or a zero gradient when grad is NULL; xnorm NULL: magnitude pruning.
cudaError_t launch_pack(const Layout& L, const RowGroups& G, const float* w, const float* xnorm,
                        const float* grad, uint4* vals, uint2* idx, uint32_t* sz, int* err,
                        cudaStream_t s);
cudaError_t launch_canon_to_device(const Layout& L, const RowGroups& G, const uint8_t* cvals,
                                   const uint8_t* cidx, const uint16_t* scale,
                                   const uint16_t* zero, uint4* vals, uint2* idx,
                                   uint32_t* sz, int* err, cudaStream_t s);
cudaError_t launch_device_to_canon(const Layout& L, const RowGroups& G, const uint4* vals,
                                   const uint2* idx, const uint32_t* sz,
                                   uint8_t* cvals, uint8_t* cidx, uint16_t* scale,
                                   uint16_t* zero, cudaStream_t s);

// ---- product kernels ----
struct RunArgs {
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  const __half* x;
  __half* y;
  int m;
  int* err;   // the handle's device error word
  int withhold = 0;   // failure-detection test hook (see sgemv_debug_withhold)
};
// Each returns cudaErrorNotSupported when it does not cover the case.
cudaError_t launch_m1(const Layout& L, const RunArgs& a, cudaStream_t s);
cudaError_t launch_mma(const Layout& L, const RunArgs& a, cudaStream_t s);
// 2 <= m <= 64 over up to 8 matrices sharing x, cols, N and m in one launch
// of the warp-level sparse MMA kernel (errors go to as[0].err).
cudaError_t launch_mma_group(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s);
// m = 1 over several matrices sharing x, cols and N in one launch.
cudaError_t launch_m1_group(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s);
// m = 1 over 2:4 matrices (L2, n2) and 1:4 matrices (L1, n1) sharing x, in
// one launch of two CTA ranges.
cudaError_t launch_m1_group_dual(const Layout* L2, const RunArgs* a2, int n2, const Layout* L1,
                                 const RunArgs* a1, int n1, cudaStream_t s);
int max_group();
// Tensor-core batch kernel (sgemv_tc.cu), 2 <= m <= 64.
size_t tc_scratch_bytes(int max_m);
int tc_tiles(const Layout& L);
bool tc_encode_weights(const Layout& L, const uint4* vals, const uint2* idx, const uint32_t* sz,
                       TcMaps* maps);
cudaError_t launch_tc(const Layout& L, const RunArgs& a, const TcMaps& maps, cudaStream_t s);
// ... on at most max_ctas CTAs (a workspace sized for that many).
cudaError_t launch_tc(const Layout& L, const RunArgs& a, const TcMaps& maps, cudaStream_t s,
                      int max_ctas);
// ... over up to tc_max_group() matrices sharing x, cols, N, the group size
// and m in one launch (partials in maps[0]'s workspace; errors to as[0].err).
int tc_max_group();
cudaError_t launch_tc_group(const Layout* Ls, const RunArgs* as, const TcMaps* const* maps,
                            int count, cudaStream_t s, int max_ctas);
// Sets the calling thread's sgemv_last_error text; returns `code`
// (report_cuda: SGEMV_ERR_CUDA with the runtime's message).
int report(int code, const char* msg);
int report_cuda(cudaError_t e, const char* what);
// Whether a product of m rows on this layout runs a kernel with the bounded
// waits that the failure-detection hook can make run out.
bool withhold_applies(const Layout& L, int m);
// Largest m that the warp-level sparse MMA kernel (sgemv_mma.cu) takes, by
// N; larger batches run the tcgen05 kernel (sgemv_tc.cu).  Measured on the
// 7B layer shapes: the mma.sp kernel is faster up to four n-tiles (m <= 32).
// 1:4 layers alone stay faster on it up to five (m <= 40), but a layer step
// that then alternates the two kernels between launches lost that gain and
// more, so both N switch at 32.
#ifndef SGEMV_MMA_MAX_M2
#define SGEMV_MMA_MAX_M2 32
#endif
#ifndef SGEMV_MMA_MAX_M1
#define SGEMV_MMA_MAX_M1 32
#endif
inline int mma_max_m(int n_keep) { return n_keep == 2 ? SGEMV_MMA_MAX_M2 : SGEMV_MMA_MAX_M1; }

}  // namespace sgemv
